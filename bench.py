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
    p.add_argument("--cpu-full", action="store_true",
                   help="also time the oracle on the whole layer once (unsampled)")
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


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, \
            "fallback"


# nominal dense tensor rates of the part (bf16 2.25 PFLOP/s, TF32 1.1 PFLOP/s): a TF32
# peak is the measured bf16 peak times their ratio
TF32_PER_BF16 = 1.1 / 2.25


def tensor_peak(peaks, clk):
    """The bf16 dense peak that applies to this run: the burst figure, unless the clocks
    sampled during the timed region show the power cap (then the sustained one)."""
    capped = "sw_power_cap" in (clk or {}).get("reasons", [])
    if capped and peaks.get("bf16_tflops_sustained"):
        return float(peaks["bf16_tflops_sustained"]), "sustained (sw_power_cap seen)"
    return float(peaks["bf16_tflops"]), "burst (no power cap seen in the timed region)"


def stage_rooflines(m, d, n, bits, w_es, block, ms, peaks, peak_src, clk, layers=1):
    """Achieved work rate of each stage of the path against the peak that bounds it.

    hessian : tensor (kind::f16), d(d+1)N flop (the lower triangle of 2 X^T X incl. the
              diagonal) per call;
    prepare : tensor (3xTF32 rank-128 updates), 2 d^3 / 3 useful flop (Cholesky plus the
              triangular inverse) against the TF32 dense peak; the panel chain (d / 128
              dependent factorizations) is reported beside it;
    quantize: HBM, per weight: read W, write and read the fp32 working copy, write E as a
              TF32 head/tail pair, write the packed codes, plus one read of U; the block
              chain (d / B dependent sweeps) beside it.
    """
    bf16, kind = tensor_peak(peaks, clk)
    tf32 = bf16 * TF32_PER_BF16
    hbm = float(peaks["hbm_gbs"])
    out = []
    h_flops = float(d) * (d + 1) * n
    a = h_flops / (ms["hessian"] / 1e3) / 1e12
    out.append({"stage": "hessian", "kernel": "hessian_tc_kernel", "bound": "tensor",
                "achieved": round(a, 3), "peak": round(bf16, 1), "unit": "TFLOP/s",
                "frac": round(a / bf16, 4), "ms": round(ms["hessian"], 4),
                "work": f"d(d+1)N = {h_flops:.4e} flop",
                "peak_source": f"{peak_src} bf16 dense, {kind}; fp16 runs at the bf16 rate"})
    p_flops = 2.0 * float(d) ** 3 / 3.0
    a = p_flops / (ms["prepare"] / 1e3) / 1e12
    panels = -(-d // 128)
    out.append({"stage": "prepare", "kernel": "potrf_kernel + rowmul_kernel + "
                "tc_gemm_short_sums_kernel (panel loop)", "bound": "tensor",
                "achieved": round(a, 3), "peak": round(tf32, 1), "unit": "TFLOP/s",
                "frac": round(a / tf32, 4), "ms": round(ms["prepare"], 4),
                "work": f"2 d^3 / 3 = {p_flops:.4e} useful flop (3xTF32 executes three TF32 "
                        f"products per useful one)",
                "peak_source": f"{peak_src} bf16 dense {kind} x 1.1/2.25 (nominal TF32:bf16)",
                "chain": {"panels": panels, "us_per_panel": round(ms["prepare"] * 1e3 / panels,
                                                                  2)}})
    q_bytes = float(m) * d * (w_es + 8 + 8 + bits / 8.0) + 4.0 * d * d
    a = q_bytes / (ms["quantize"] / 1e3) / 1e9
    blocks = -(-d // block)
    pairs = -(-blocks // 2) if block > 1 else blocks
    out.append({"stage": "quantize", "kernel": ("grid_kernel + sweep_pair_kernel + "
                "tc_gemm_one_sum_kernel + pack_kernel") if block > 1 else
                "grid_kernel + eager_column_kernel + pack_kernel", "bound": "hbm",
                "achieved": round(a, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(a / hbm, 4), "ms": round(ms["quantize"], 4),
                "work": f"{q_bytes:.4e} bytes: per weight W read ({w_es} B), fp32 working "
                        f"copy written and read (8 B), E head/tail written (8 B), packed "
                        f"codes ({bits / 8:g} B); U read once (4 d^2 B)",
                "peak_source": f"{peak_src} copy bandwidth",
                "chain": ({"pairs of blocks": pairs,
                           "us_per_pair": round(ms["quantize"] * 1e3 / pairs, 2)} if block > 1
                          else {"columns": blocks,
                                "us_per_column": round(ms["quantize"] * 1e3 / blocks, 2)})})
    if layers != 1:
        for r in out:
            r["layers"] = layers
    return out


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

def oracle_group_sample(X_rows, layers, n_tok, d, bits_list, block, damp):
    """Times the fp64 oracle on a bounded sample of one input group of a workload (its
    Hessian and prepare once, the sweep of each of its layers at each bit width) and scales
    each stage by its operation count to the whole group.

    X_rows: ``[t, c]`` float32 token-major inputs drawn by the group's recipe (t <= n_tok
    tokens, c <= d channels); ``layers``: ``(W_sample [r, c] float32, d_out)`` per layer.
    Hessian x (n_tok / t)(d / c)^2, prepare x (d / c)^3, each sweep x (d_out / r)(d / c)^2.
    Returns ``(measured_s, estimated_full_s, detail)``.
    """
    from oracle import gptq_oracle as O
    t, c = X_rows.shape
    t0 = time.perf_counter()
    H = O.hessian(X_rows)
    t1 = time.perf_counter()
    Hd, dead, _ = O.damp_hessian(H, damp)
    U = O.inverse_cholesky_upper(Hd)
    t2 = time.perf_counter()
    f_h, f_p = (n_tok / t) * (d / c) ** 2, (d / c) ** 3
    meas, est = t2 - t0, (t1 - t0) * f_h + (t2 - t1) * f_p
    sweeps = []
    for Ws, m in layers:
        for b in bits_list:
            t3 = time.perf_counter()
            scale, zero = O.row_grid(Ws, b)
            codes, _ = O.gptq_quantize(Ws, U, scale, zero, b, block=block, dead=dead)
            O.pack_codes(codes, b)
            dt = time.perf_counter() - t3
            f_q = (m / Ws.shape[0]) * (d / c) ** 2
            meas += dt
            est += dt * f_q
            sweeps.append({"rows": int(Ws.shape[0]), "bits": b, "sweep_s": dt, "scale": f_q})
    detail = {"hessian_s": t1 - t0, "prepare_s": t2 - t1, "tokens": t, "channels": c,
              "scale": {"hessian": f_h, "prepare": f_p}, "sweeps": sweeps}
    return meas, est, detail


def sample_text(det):
    sw = det["sweeps"]
    return (f"fp64 NumPy oracle on a sample, each stage scaled by its operation count: "
            f"Hessian over {det['tokens']} tokens x {det['channels']} channels "
            f"(x{det['scale']['hessian']:.3g}), prepare at {det['channels']} channels "
            f"(x{det['scale']['prepare']:.3g}), {len(sw)} sweep(s) of {sw[0]['rows']} rows "
            f"(x{sw[0]['scale']:.3g})")


def oracle_layer_unsampled(X_chunk, W, n_tok, bits, block, damp):
    """The fp64 oracle on a whole layer, timed once: the Hessian accumulated over n_tok
    tokens in passes over the given token chunk (the fp64 products take the same time
    whatever the values), the prepare and the sweep of every row at full width."""
    from oracle import gptq_oracle as O
    t0 = time.perf_counter()
    H = None
    done = 0
    while done < n_tok:
        take = min(X_chunk.shape[0], n_tok - done)
        H = O.hessian(X_chunk[:take], H)
        done += take
    t1 = time.perf_counter()
    Hd, dead, _ = O.damp_hessian(H, damp)
    U = O.inverse_cholesky_upper(Hd)
    t2 = time.perf_counter()
    scale, zero = O.row_grid(W, bits)
    codes, _ = O.gptq_quantize(W, U, scale, zero, bits, block=block, dead=dead)
    O.pack_codes(codes, bits)
    t3 = time.perf_counter()
    return {"seconds": t3 - t0, "hessian_s": t1 - t0, "prepare_s": t2 - t1,
            "sweep_s": t3 - t2, "tokens": n_tok, "chunk_tokens": int(X_chunk.shape[0])}


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
    w_es = 2 if layer.w_dtype in ("bf16", "f16") else 4
    stages = stage_rooflines(m, d, n, bits, w_es, block,
                             {"hessian": st_h, "prepare": st_p, "quantize": st_q},
                             peaks, peak_src, clk)
    # the dominant kernel: the Hessian's one launch per step (its stage time is that launch,
    # timed by events on the stream it runs on); with B = 1 the eager column updates
    roofline = dict(stages[0])
    roofline["kernel"] = "hessian_tc_kernel (gptq_hessian_accumulate: one launch per step)"
    roofline["traffic"] = None
    roofline["traffic_note"] = ("not measured in this run (ncu does not run inside the bench): "
                                "the DRAM bytes of an ncu capture of this kernel, scaled to this "
                                "launch, are stated with its profile summary")
    if block == 1:
        # the eager sweep dominates (B = 1): each column's update reads and writes the fp32
        # working copy of every later column once
        q_bytes = float(sum(m * (d - j - 1) * 8 for j in range(d)))
        q_gbs = q_bytes / (st_q / 1e3) / 1e9
        roofline = {"kernel": "eager_column_kernel (quantize stage, one launch per column)",
                    "bound": "hbm", "achieved": round(q_gbs, 1), "peak": float(peaks["hbm_gbs"]),
                    "unit": "GB/s", "frac": round(q_gbs / float(peaks["hbm_gbs"]), 4),
                    "traffic": None,
                    "algorithmic": f"sum over columns of d_out*(d_in - j - 1)*8 bytes = "
                                   f"{q_bytes:.4e} per layer (fp32 read + write of the later "
                                   f"columns per column)",
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
        c = min(d, 4096)
        Xs = X[:min(n, 16384), :c].float().cpu().numpy()
        Ws = W[:min(m, 1024), :c].float().cpu().numpy()
        meas, est, det = oracle_group_sample(Xs, [(Ws, m)], n, d, (bits,), block, damp)
        cpu = {"value": weights / est, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
               "sample": sample_text(det), "measured_s": meas, "est_seconds_per_layer": est,
               "detail": det}
        if args.cpu_full:
            cpu["unsampled"] = oracle_layer_unsampled(X[:16384].float().cpu().numpy(),
                                                      W.float().cpu().numpy(), n, bits,
                                                      block, damp)

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
            # the quantize-only time (dead columns and damping through packing, the Hessian
            # left out: it is usually spread over the calibration passes)
            "quantize_only": {"ms": st_p + st_q, "unit": UNIT,
                              "value": whole_job_value(weights, world, st_p + st_q)},
            "roofline": roofline, "roofline_stages": stages, "cpu_baseline": cpu, "e2e": e2e,
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
    peak_t, peak_kind = tensor_peak(peaks, clk)
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
                     "peak_source": f"{peak_src} bf16 dense, {peak_kind}; fp16 runs at the "
                                    f"bf16 rate"},
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
    peak_t, peak_kind = tensor_peak(peaks, clk)
    # every stage of the serialized pass against its bound (work summed over groups, layers
    # and bit widths)
    p_flops = float(sum(2.0 * x.shape[1] ** 3 / 3.0 for x, _ in G))
    q_bytes = float(sum(len(wl.bits) * (W.shape[0] * W.shape[1] * (W.element_size() + 16)
                                        + sum(W.shape[0] * W.shape[1] * b / 8.0
                                              for b in wl.bits) / len(wl.bits))
                        + len(wl.bits) * 4.0 * x.shape[1] ** 2
                        for x, Ws in G for W in Ws))
    tf32 = peak_t * TF32_PER_BF16
    hbm = float(peaks["hbm_gbs"])
    p_tf = p_flops / (stages["prepare"] / 1e3) / 1e12
    q_gbs = q_bytes / (stages["quantize"] / 1e3) / 1e9
    stage_list = [
        {"stage": "hessian", "bound": "tensor", "achieved": round(h_tf, 3),
         "peak": round(peak_t, 1), "unit": "TFLOP/s", "frac": round(h_tf / peak_t, 4),
         "ms": round(stages["hessian"], 4), "work": f"sum d(d+1)N = {h_flops:.4e} flop"},
        {"stage": "prepare", "bound": "tensor", "achieved": round(p_tf, 3),
         "peak": round(tf32, 1), "unit": "TFLOP/s", "frac": round(p_tf / tf32, 4),
         "ms": round(stages["prepare"], 4),
         "work": f"sum 2 d^3 / 3 = {p_flops:.4e} useful flop (3xTF32)",
         "peak_source": "bf16 peak x 1.1/2.25 (nominal TF32:bf16)"},
        {"stage": "quantize", "bound": "hbm", "achieved": round(q_gbs, 1), "peak": hbm,
         "unit": "GB/s", "frac": round(q_gbs / hbm, 4), "ms": round(stages["quantize"], 4),
         "work": f"{q_bytes:.4e} bytes (per weight and bit width: W read, fp32 working copy "
                 f"written and read, E head/tail written, packed codes; U read per sweep)"}]
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
                     "peak_source": f"{peak_src} bf16 dense, {peak_kind}"},
        "roofline_stages": stage_list,
        "gpu_launches": int(launches), "clocks": clk,
    }
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference(args, rank, world):
    """The fp64 oracle on the host cores.  Each step times a bounded sample of the workload
    (every stage of every layer, drawn by the workload's recipe at the sample's size) and
    scales each stage by its operation count to the whole workload; ``ms_per_step`` is the
    measured time of the sample, ``value`` the whole-workload rate it implies.  A
    single-layer workload of at most 4096 channels is also timed once unsampled, outside
    the step loop.  Under torchrun only rank 0 runs."""
    if rank != 0:
        return
    from post_weight_quantization_03_gb300 import synthetic as S
    from dataclasses import replace

    wl = S.WORKLOADS[args.workload]
    block = args.block or wl.block
    if args.obq:
        return run_reference_obq(args, world)
    groups = {}
    for layer in wl.layers:
        groups.setdefault(layer.act, []).append(layer)
    samples = []
    for act, layers in groups.items():
        n = args.n_tok or act.n_tok
        c = min(act.d_in, 4096)
        t = min(n, 16384)
        Xs = S.activations(replace(act, d_in=c, n_dead=min(act.n_dead, c // 100),
                                   n_outlier=min(act.n_outlier, c // 100)), device="cpu",
                           n_tok=t).float().numpy()
        Ls = [(S.weights(min(l.d_out, 1024), c, l.w_std, l.w_dtype,
                         l.act.seed * 131 + l.w_seed).float().numpy(), l.d_out) for l in layers]
        samples.append((Xs, Ls, n, act.d_in))
    bits_list = wl.bits if len(wl.layers) > 1 else (wl.bits[-1],)
    weights = sum(l.d_out * l.act.d_in for l in wl.layers) * len(bits_list)
    unsampled = None
    if len(wl.layers) == 1 and wl.layers[0].act.d_in <= 4096:
        layer = wl.layers[0]
        Xs, Ls, n, d = samples[0]
        Wfull = S.layer_weights(layer).float().numpy()
        unsampled = oracle_layer_unsampled(Xs, Wfull, n, bits_list[0], block, wl.damp)
        unsampled["value"] = weights / unsampled["seconds"]
    meas, ests, dets = [], [], []
    for i in range(args.warmup + args.steps):
        m_t, e_t, d_all = 0.0, 0.0, []
        for Xs, Ls, n, d in samples:
            mt, et, det = oracle_group_sample(Xs, Ls, n, d, bits_list, block, wl.damp)
            m_t += mt
            e_t += et
            d_all.append(det)
        if i >= args.warmup:
            meas.append(m_t)
            ests.append(e_t)
            dets = d_all
    est = statistics.mean(ests)
    value = weights / est
    sample = "; ".join(sample_text(dt) for dt in dets)
    cpu = {"value": value, "unit": UNIT, "cores": host_cores(), "kind": "oracle",
           "sample": sample, "est_seconds_per_workload": est}
    if unsampled is not None:
        cpu["unsampled"] = unsampled
    out = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": statistics.mean(meas) * 1e3,
           "ms_per_layer_est": est * 1e3 / len(wl.layers) / len(bits_list),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
           "data": "synthetic", "impl": "reference",
           "config": {"workload": wl.name, "layers": [l.name for l in wl.layers],
                      "bits": list(bits_list), "block": block, "damp": wl.damp},
           "cpu_baseline": cpu,
           "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0},
           "detail": dets}
    print(json.dumps(out), flush=True)


def run_reference_obq(args, world):
    """The oracle's greedy-order OBQ on rows of the 4096 x 128 layer, scaled to all rows."""
    from oracle import gptq_oracle as O
    from post_weight_quantization_03_gb300 import synthetic as S
    m, d, bits = 4096, 128, 4
    n = args.n_tok or 65536
    act = S.ActivationSpec(d_in=d, n_tok=n, dtype="f16", n_dead=2, n_outlier=2, seed=77)
    X = S.activations(act, device="cpu").float().numpy()
    W = S.weights(m, d, 0.02, "bf16", 78).float().numpy()
    Hd, dead, _ = O.damp_hessian(O.hessian(X), 0.01)
    rows = 64
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        s_, z_ = O.row_grid(W[:rows], bits)
        O.obq_greedy(W[:rows], Hd, s_, z_, bits, dead=dead)
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    sec = statistics.mean(times) * m / rows
    value = m * d / sec
    out = {"metric": "ms per layer: OBQ greedy order vs fixed-order GPTQ (4096 x 128 int4)",
           "value": value, "unit": "weights/s", "n_gpus": world, "steps": args.steps,
           "warmup": args.warmup, "ms_per_step": statistics.mean(times) * 1e3,
           "ms_per_layer_est": sec * 1e3, "higher_is_better": True, "scaling": "weak",
           "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
           "config": {"workload": "obq4096x128", "d_out": m, "d_in": d, "n_tok": n,
                      "bits": bits},
           "cpu_baseline": {"value": value, "unit": "weights/s", "cores": host_cores(),
                            "kind": "oracle",
                            "sample": f"fp64 NumPy OBQ oracle on {rows} rows, x{m // rows}"},
           "e2e": {"value": value, "unit": "weights/s", "h2d_bytes_per_step": 0,
                   "d2h_bytes_per_step": 0}}
    print(json.dumps(out), flush=True)


if __name__ == "__main__":
    main()
