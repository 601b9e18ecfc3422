"""Benchmark of the NVFP4 linear-layer hot path on GB300.

One step = one NVFP4 linear layer forward + backward at the 12B model's FFN
up-projection shape (M = 8192 tokens, N = 20480, K = 5120), through the C ABI:
  Fprop : amax + 1x16 RTN quantize of X; amax + 16x16 RTN quantize of W (both
          layouts); GEMM Y = Xq Wq^T (bf16 out)
  Dgrad : amax + 1x16 SR quantize of dY; GEMM dX = dYq Wq (bf16 out)
  Wgrad : RHT amax + RHT 1x16 SR colwise quantize of dY; RHT amax + RHT RTN
          colwise quantize of X; GEMM dW = (H dY)^T (H X) (fp32 out)
value = GEMM FLOPs of the step (3 x 2MNK) / step time (quantization included).

Usage: python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
With N > 1 (launched by torchrun) every rank runs an independent replica of
the step (weak scaling); rank 0 prints the JSON line.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import tempfile
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

M, N, K = 8192, 20480, 5120
METRIC = "NVFP4 GEMM TFLOPS (8192x20480x5120) and quantize+RHT GB/s vs roofline"
UNIT = "TFLOP/s"
WORKLOAD = ("NVFP4 linear layer fwd+bwd (Fprop+Dgrad+Wgrad GEMMs with all quantizations), "
            "X 8192x5120, W 20480x5120, dY 8192x20480 bf16; 12B hybrid model FFN up-projection at seq 8192")
FP4_OVER_BF16 = 13.5 / 2.25       # nominal dense FP4 / BF16 tensor rate on GB300
FALLBACK_HBM_GBS, FALLBACK_BF16_TFLOPS = 6800.0, 1900.0
L2_FLUSH_BYTES = 256 << 20


def _env_rank():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), \
        int(os.environ.get("LOCAL_RANK", "0"))


def max_over_ranks(value: float, device=None) -> float:
    """Max of a per-rank float over all ranks (identity when not distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device or "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def _peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        p = json.load(open(path))
        return dict(hbm=float(p["hbm_gbs"]), bf16=float(p["bf16_tflops"]),
                    bf16_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])), source="measured")
    return dict(hbm=FALLBACK_HBM_GBS, bf16=FALLBACK_BF16_TFLOPS, bf16_sustained=1700.0, source="fallback")


# ---- profile summaries: DRAM traffic of the dominant kernel ------------------------

def _profile_traffic(summary: str, sources: tuple, field: str):
    """DRAM bytes from a committed ncu summary (its `field` line), or None if
    the summary is missing or any of the kernel sources it was taken on
    (its `source_sha256 <file>: <hash>` lines) has changed since."""
    path = os.path.join(ROOT, "profiles", summary)
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and not line.startswith(" "):
            k, v = line.split(":", 1)
            fields[k.strip()] = v.strip()
    for name in sources:
        src = open(os.path.join(ROOT, "quantize_block_scaled_amax_gb300", "csrc", name), "rb").read()
        if fields.get(f"source_sha256 {name}", "") != hashlib.sha256(src).hexdigest():
            return None
    try:
        return float(fields[field])
    except (KeyError, ValueError):
        return None


# ---- clocks ---------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = open(self._path(), "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def _path(self):
        # the raw samples; the JSON line carries their summary
        d = os.environ.get("BENCH_CLOCKS_DIR") or tempfile.gettempdir()
        return os.path.join(d, f"bench_clocks_{os.getpid()}.csv")

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.close()
        rows = []
        for line in open(self._path()):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append(dict(sm=float(parts[1]), max=float(parts[2]), power=float(parts[3]), active=parts[4],
                                 hw=parts[5], hw_thermal=parts[6], sw_thermal=parts[7], sw_power=parts[8]))
            except ValueError:
                continue
        if not rows:
            return None
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hw_thermal", "hw_thermal_slowdown"),
                              ("sw_thermal", "sw_thermal_slowdown"), ("sw_power", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows), "sm_max_mhz": max(r["max"] for r in rows),
                "power_w_max": max(r["power"] for r in rows), "samples": len(rows), "reasons": sorted(reasons)}


# ---- the GPU step -------------------------------------------------------------------

def gpu_bench(args):
    import torch
    import torch.distributed as dist

    rank, world, local_rank = _env_rank()
    if world > 1:
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    dev = torch.device("cuda", torch.cuda.current_device())

    from quantize_block_scaled_amax_gb300 import build as _b
    _b.build()
    import quantize_block_scaled_amax_gb300 as nv
    import workloads

    x = workloads.activations(M, K, device=dev)
    w = workloads.weights(N, K, device=dev)
    dy = workloads.gradients(M, N, device=dev)
    ctx = nv.LinearContext(M, N, K, dev)
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(N, K, dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED

    # the step, op by op through the C ABI (the same calls nvfp4_linear_fwd_rht
    # and nvfp4_linear_bwd with X = NULL make)
    ops = [
        # X rowwise (Fprop) and RHT colwise (Wgrad), RTN, both tensor amaxes from one read
        ("quant_x_rtn_and_rht", lambda: nv.nvfp4_quantize_with_rht(x, round="rtn", rht_seed=rh, out_rowwise=ctx.xq,
                                                                     out_colwise=ctx.xtq)),
        ("quant_w_16x16_both", lambda: nv.nvfp4_quantize(w, block="16x16", colwise=True, out_rowwise=ctx.wq,
                                                         out_colwise=ctx.wtq)),
        ("gemm_fprop", lambda: nv.nvfp4_gemm(ctx.xq, ctx.wq, out=y)),
        # dY rowwise (Dgrad) and RHT colwise (Wgrad), SR, both tensor amaxes from one read
        ("quant_dy_sr_and_rht", lambda: nv.nvfp4_quantize_with_rht(dy, round="sr", seed=sr, rht_seed=rh,
                                                                     out_rowwise=ctx.dyq, out_colwise=ctx.dytq)),
        ("gemm_dgrad", lambda: nv.nvfp4_gemm(ctx.dyq, ctx.wtq, out=dx)),
        ("gemm_wgrad", lambda: nv.nvfp4_gemm(ctx.dytq, ctx.xtq, out=dw)),
    ]
    launches_per_op = {"quant_x_rtn_and_rht": 3, "quant_w_16x16_both": 2, "gemm_fprop": 1, "quant_dy_sr_and_rht": 3,
                       "gemm_dgrad": 1, "gemm_wgrad": 1}
    # algorithmic bytes: the amax pass reads the input once, the encode pass
    # reads it again and writes codes (1/2 byte per element) and one E4M3
    # scale per 16 elements per layout
    bx, bw, bdy = M * K * 2, N * K * 2, M * N * 2
    op_bytes = {
        # one amax read, two encode reads, codes and scales of both layouts
        "quant_x_rtn_and_rht": 3 * bx + 2 * (M * K // 2 + M * K // 16),
        "quant_w_16x16_both": 2 * bw + 2 * (N * K // 2 + N * K // 16),
        "quant_dy_sr_and_rht": 3 * bdy + 2 * (M * N // 2 + M * N // 16),
    }
    gemm_flops = 2.0 * M * N * K

    stream = torch.cuda.current_stream()
    for _ in range(args.warmup):
        for _, fn in ops:
            fn()
    torch.cuda.synchronize()
    st = nv.nvfp4_sync_status()
    if st != nv.OK:
        raise RuntimeError(f"device status {st} after warm-up")

    # The timed step: the layer's two public calls, nvfp4_linear_fwd_rht (X
    # and X^T's RHT codes from one amax read, W's 16x16 codes on the
    # library's second stream meanwhile, Fprop) and nvfp4_linear_bwd with
    # X = NULL (dY's SR codes, Dgrad, Wgrad): the same launches as the op list.
    def layer_step():
        nv.nvfp4_linear_fwd(x, w, ctx, Y=y, rht_seed=rh)
        nv.nvfp4_linear_bwd(dy, None, ctx, sr_seed=sr, rht_seed=rh, dX=dx, dW=dw)

    for _ in range(args.warmup):
        layer_step()
    torch.cuda.synchronize()
    step_evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                for _ in range(args.steps)]
    sampler = ClockSampler(dev.index)
    if rank == 0:
        sampler.start()
        time.sleep(0.3)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    for s in range(args.steps):
        flush.fill_(s & 0xFF)                  # evict L2 between steps (not timed)
        step_evs[s][0].record(stream)
        layer_step()
        step_evs[s][1].record(stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop() if rank == 0 else None
    st = nv.nvfp4_sync_status()
    if st != nv.OK:
        raise RuntimeError(f"device status {st} after the timed steps")
    ms_per_step = max_over_ranks(sum(a.elapsed_time(b) for a, b in step_evs), dev) / args.steps
    value = world * 3 * gemm_flops / (ms_per_step * 1e-3) / 1e12

    # The same step op by op (one stream, an event pair around each op) for
    # the per-kernel times, rooflines and shares.
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in ops]
           for _ in range(args.steps)]
    torch.cuda.synchronize()
    for s in range(args.steps):
        flush.fill_(s & 0xFF)
        for (name, fn), (e0, e1) in zip(ops, evs[s]):
            e0.record(stream)
            fn()
            e1.record(stream)
    torch.cuda.synchronize()
    per_op = {name: 0.0 for name, _ in ops}
    for s in range(args.steps):
        for (name, _), (e0, e1) in zip(ops, evs[s]):
            per_op[name] += e0.elapsed_time(e1)
    ops_ms_per_step = max_over_ranks(sum(per_op.values()), dev) / args.steps

    # ---- end to end: host buffers in, results back, through nvfp4_linear_fwd_rht/bwd.
    # Every step copies its inputs X, W, dY from pinned host memory and its
    # results Y, dX, dW back.  The copies run on their own streams (one per
    # direction) and device buffers are double-buffered, so step i's results
    # go back while step i+1 computes, as a training loop's data movement
    # would; the compute itself stays on one stream.
    e2e = None
    if not args.no_e2e:
        xh = x.cpu().pin_memory()
        wh = w.cpu().pin_memory()
        dyh = dy.cpu().pin_memory()
        yh = torch.empty(M, N, dtype=torch.bfloat16).pin_memory()
        dxh = torch.empty(M, K, dtype=torch.bfloat16).pin_memory()
        dwh = torch.empty(N, K, dtype=torch.float32).pin_memory()
        din = [(torch.empty_like(x), torch.empty_like(w), torch.empty_like(dy)) for _ in range(2)]
        dout = [(torch.empty_like(y), torch.empty_like(dx), torch.empty_like(dw)) for _ in range(2)]
        h2d, d2h = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        ev = {k: [torch.cuda.Event() for _ in range(2)] for k in ("xw", "dy", "y", "bwd", "in_free", "out_free")}

        def e2e_step(i):
            b = i % 2
            xd, wd, dyd = din[b]
            yd, dxd, dwd = dout[b]
            with torch.cuda.stream(h2d):
                if i >= 2:
                    h2d.wait_event(ev["in_free"][b])
                xd.copy_(xh, non_blocking=True)
                wd.copy_(wh, non_blocking=True)
                ev["xw"][b].record(h2d)
                dyd.copy_(dyh, non_blocking=True)
                ev["dy"][b].record(h2d)
            stream.wait_event(ev["xw"][b])
            if i >= 2:
                stream.wait_event(ev["out_free"][b])
            nv.nvfp4_linear_fwd(xd, wd, ctx, Y=yd, rht_seed=rh)       # also X^T's Wgrad codes
            ev["y"][b].record(stream)
            stream.wait_event(ev["dy"][b])
            nv.nvfp4_linear_bwd(dyd, None, ctx, sr_seed=sr, rht_seed=rh, dX=dxd, dW=dwd)
            ev["bwd"][b].record(stream)
            ev["in_free"][b].record(stream)
            with torch.cuda.stream(d2h):
                d2h.wait_event(ev["y"][b])
                yh.copy_(yd, non_blocking=True)
                d2h.wait_event(ev["bwd"][b])
                dxh.copy_(dxd, non_blocking=True)
                dwh.copy_(dwd, non_blocking=True)
                ev["out_free"][b].record(d2h)

        for i in range(2):
            e2e_step(i)
        torch.cuda.synchronize()
        e_steps = max(4, args.steps // 4)
        a, b_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        h2d.wait_event(a)
        for i in range(e_steps):
            e2e_step(i)
        stream.wait_event(ev["out_free"][(e_steps - 1) % 2])
        b_end.record(stream)
        torch.cuda.synchronize()
        e2e_ms = max_over_ranks(a.elapsed_time(b_end) / e_steps, dev)
        e2e = {"value": round(world * 3 * gemm_flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": UNIT,
               "ms_per_step": round(e2e_ms, 4),
               "h2d_bytes_per_step": int(xh.numel() * 2 + wh.numel() * 2 + dyh.numel() * 2),
               "d2h_bytes_per_step": int(yh.numel() * 2 + dxh.numel() * 2 + dwh.numel() * 4),
               "api": "nvfp4_linear_fwd_rht + nvfp4_linear_bwd with pinned host buffers; copies on one stream per "
                      "direction, device buffers double-buffered so copies overlap the neighbouring steps' compute"}
    st = nv.nvfp4_sync_status()
    if st != nv.OK:
        raise RuntimeError(f"device status {st} after the timed region")

    mx = None if args.no_mx else mx_measure(nv, x, w, dy, flush, stream, max(5, args.steps // 10))
    rht_rows = None if args.no_mx else rht_rows_measure(nv, x, w, dy, flush, stream, max(5, args.steps // 10))
    bf16_gemm = None if args.no_mx else bf16_gemm_measure(nv, x, w, flush, stream, max(5, args.steps // 10),
                                                          _peaks())
    ffn = None if args.no_ffn else ffn_measure(nv, flush, stream, max(5, args.steps // 4), _peaks())

    if rank != 0:
        if world > 1:
            dist.barrier()
            dist.destroy_process_group()
        return None

    peaks = _peaks()
    # each GEMM is event-timed on its own, a fraction of a millisecond: the
    # burst figure applies
    fp4_peak = peaks["bf16"] * FP4_OVER_BF16
    kernels = {}
    for name, ms in per_op.items():
        avg = ms / args.steps
        if name.startswith("gemm"):
            ach = gemm_flops / (avg * 1e-3) / 1e12
            kernels[name] = {"ms": round(avg, 4), "tflops": round(ach, 1), "frac": round(ach / fp4_peak, 4)}
        else:
            ach = op_bytes[name] / (avg * 1e-3) / 1e9
            kernels[name] = {"ms": round(avg, 4), "gbs": round(ach, 1), "frac": round(ach / peaks["hbm"], 4),
                             "bytes": op_bytes[name]}
    gemm_ms = sum(v["ms"] for k, v in kernels.items() if k.startswith("gemm"))
    quant_ms = sum(v["ms"] for k, v in kernels.items() if not k.startswith("gemm"))
    quant_bytes = sum(op_bytes.values())
    quant_gbs = quant_bytes / (quant_ms * 1e-3) / 1e9
    gemm_avg_ms = gemm_ms / 3
    gemm_ach = gemm_flops / (gemm_avg_ms * 1e-3) / 1e12
    roof_gemm = {"bound": "tensor", "achieved": round(gemm_ach, 1), "peak": round(fp4_peak, 1), "unit": "TFLOP/s",
                 "frac": round(gemm_ach / fp4_peak, 4),
                 # DRAM bytes per launch (ncu, average of the three GEMM launches)
                 "traffic": _profile_traffic("gemm_nvf4_layer_gemms_dram_8192x20480x5120.txt", ("gemm.cu",),
                                             "dram_bytes_per_launch_full_size"),
                 "kernel": "nvf4_gemm_kernel (avg of Fprop, Dgrad, Wgrad launches)",
                 "peak_source": f"{peaks['source']} burst bf16 {peaks['bf16']} TFLOP/s x "
                                f"{FP4_OVER_BF16:g} (nominal FP4/BF16 ratio)"}
    # DRAM bytes of all the step's quantize launches (ncu, cold cache per kernel)
    quant_traffic = _profile_traffic("quantize_step_dram_8192x20480x5120.txt", ("quantize.cu", "nvfp4_device.cuh"),
                                     "dram_bytes_per_step")
    roof_quant = {"bound": "hbm", "achieved": round(quant_gbs, 1), "peak": peaks["hbm"], "unit": "GB/s",
                  "frac": round(quant_gbs / peaks["hbm"], 4), "traffic": quant_traffic,
                  "traffic_unit": "bytes per step (all quantize launches)",
                  "kernel": "all quantize + RHT launches of the step (amax pass + encode pass)",
                  "peak_source": f"{peaks['source']} HBM copy bandwidth"}
    dominant_is_gemm = gemm_ms >= quant_ms
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "ms_per_step_ops": round(ops_ms_per_step, 4),
        "vs_baseline": None, "dtype": "nvfp4 (e2m1 x e2m1, e4m3 block scales, fp32 accumulate; fp32 quantize)",
        "data": "synthetic (seeded: X N(0,1)+0.1% x50 outliers, W N(0,0.02), dY Student-t(3)*1e-3)",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "l2": "flushed between steps (256 MB write)",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "quantize_rht_gbs": round(quant_gbs, 1),
        "gemm_tflops": round(gemm_ach, 1),
        "roofline": roof_gemm if dominant_is_gemm else roof_quant,
        "roofline_quantize": roof_quant,
        "roofline_gemm": roof_gemm,
        "kernels": kernels,
        "share": {"gemm": round(gemm_ms / (gemm_ms + quant_ms), 4), "quantize": round(quant_ms / (gemm_ms + quant_ms), 4)},
        # the timed steps: the op list's launches, Dgrad and Wgrad being one
        # launch in nvfp4_linear_bwd (nvfp4_gemm_pair)
        "gpu_launches": args.steps * (sum(launches_per_op.values()) - 1),
        "gpu_launches_per_step_ops": sum(launches_per_op.values()),
        "mxfp4": mx,
        "rht_fprop_dgrad_quantize": rht_rows,
        "bf16_fallback_gemm": bf16_gemm,
        "ffn": ffn,
        "e2e": e2e,
        "clocks": clocks,
    }
    if not args.no_cpu_baseline:
        out["cpu_baseline"] = cpu_baseline_subprocess(args.cpu_sample_m, args.cpu_sample_n)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    return out


# ---- the oracle on the host cores ----------------------------------------------------

def oracle_inputs(m: int, n: int, k: int):
    """Seeded inputs of a bounded sample of the layer: m tokens, n output
    features, the full K."""
    import workloads
    x = workloads.activations(m, k, seed=workloads.SEED_BASE + 10).float().numpy()
    w = workloads.weights(n, k, seed=workloads.SEED_BASE + 11).float().numpy()
    dy = workloads.gradients(m, n, seed=workloads.SEED_BASE + 12).float().numpy()
    return x, w, dy


def oracle_step(x, w, dy):
    """The step computed by the oracle: every quantization of the recipe and
    the three GEMMs (FP64 products of the dequantized operands)."""
    import numpy as np
    import oracle
    import workloads

    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    qx = oracle.quantize(x)
    qw = oracle.quantize(w, block="16x16")
    qwt = oracle.quantize(w, layout="col", block="16x16")
    y = oracle.gemm(qx, qw)
    qdy = oracle.quantize(dy, rounding="sr", seed=sr)
    dx = oracle.gemm(qdy, qwt)
    qdyt = oracle.quantize(dy, layout="col", rounding="sr", seed=sr, rht_seed=rh)
    qxt = oracle.quantize(x, layout="col", rht_seed=rh)
    dw = oracle.gemm(qdyt, qxt)
    return float(np.abs(y).sum() + np.abs(dx).sum() + np.abs(dw).sum())


def _oracle_sample_desc(m, n):
    return (f"oracle step on a {m}-token x {n}-feature slice of the layer at K={K} "
            f"(quantize X, W 16x16 both layouts, dY SR, RHT dY^T SR, RHT X^T; Fprop, Dgrad, Wgrad FP64 GEMMs); "
            f"value = 3*2*{m}*{n}*{K} FLOP / oracle time")


def _host_cores() -> int:
    return len(os.sched_getaffinity(0))


def cpu_baseline_subprocess(m: int, n: int):
    """Time the oracle in fresh processes (none forked after CUDA): on all
    host cores over the full step (every quantization in full, the GEMMs on
    sampled output rows, extrapolated), and on one core over a slice."""
    out = {}
    for mode, threads in (("full", _host_cores()), ("slice", 1)):
        env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
                   MKL_NUM_THREADS=str(threads), CUDA_VISIBLE_DEVICES="")
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--cpu-baseline-only", mode, "--cpu-sample-m",
                            str(m), "--cpu-sample-n", str(n)], capture_output=True, text=True, env=env, timeout=1800)
        if r.returncode != 0:
            out[mode] = {"error": r.stderr.strip().splitlines()[-1] if r.stderr.strip() else f"rc {r.returncode}"}
        else:
            out[mode] = json.loads(r.stdout.strip().splitlines()[-1])
    res = dict(out["full"])
    res["single_core"] = out["slice"]
    return res


def _timed(fn):
    t0 = time.perf_counter()
    r = fn()
    return r, time.perf_counter() - t0


def cpu_baseline_only(mode: str, m: int, n: int):
    import torch
    threads = int(os.environ.get("OMP_NUM_THREADS", "1"))
    torch.set_num_threads(threads)
    import oracle
    oracle.build()
    oracle_step(*oracle_inputs(16, 64, K))          # load and warm the library
    if mode == "slice":
        inputs = oracle_inputs(m, n, K)
        _, dt = _timed(lambda: oracle_step(*inputs))
        flops = 3 * 2.0 * m * n * K
        print(json.dumps({"value": round(flops / dt / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
                          "seconds": round(dt, 3), "sample": _oracle_sample_desc(m, n)}))
        return
    # full: the oracle on the whole layer step, every quantization in full;
    # each GEMM's dequantized B operand in full and 256 sampled output rows,
    # its row time extrapolated linearly to all rows
    import numpy as np
    import workloads
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    x = workloads.activations(M, K).float().numpy()
    w = workloads.weights(N, K).float().numpy()
    dy = workloads.gradients(M, N).float().numpy()
    t_quant = 0.0
    q = {}
    for name, fn in (("x", lambda: oracle.quantize(x)),
                     ("w", lambda: oracle.quantize(w, block="16x16")),
                     ("wt", lambda: oracle.quantize(w, layout="col", block="16x16")),
                     ("dy", lambda: oracle.quantize(dy, rounding="sr", seed=sr)),
                     ("dyt", lambda: oracle.quantize(dy, layout="col", rounding="sr", seed=sr, rht_seed=rh)),
                     ("xt", lambda: oracle.quantize(x, layout="col", rht_seed=rh))):
        q[name], dt = _timed(fn)
        t_quant += dt
    rows = 256
    t_gemm_est = 0.0
    for a, b in (("x", "w"), ("dy", "wt"), ("dyt", "xt")):
        bd, t_b = _timed(lambda: oracle.dequantize(q[b]))
        qa = dict(q[a], codes=q[a]["codes"][:rows], scales=q[a]["scales"][:rows])
        _, t_rows = _timed(lambda: oracle.dequantize(qa) @ bd.T)
        t_gemm_est += t_b + t_rows * q[a]["codes"].shape[0] / rows
        del bd
    est = t_quant + t_gemm_est
    flops = 3 * 2.0 * M * N * K
    print(json.dumps({
        "value": round(flops / est / 1e12, 6), "unit": UNIT, "cores": threads, "kind": "oracle",
        "seconds": round(est, 3), "seconds_quantize_measured": round(t_quant, 3),
        "seconds_gemm_extrapolated": round(t_gemm_est, 3),
        "sample": (f"oracle on the full layer step M={M} N={N} K={K}: all six quantizations of the recipe in full "
                   f"(measured); the three FP64 GEMMs on {rows} sampled output rows each plus the dequantized B "
                   f"operand, row time extrapolated linearly to all rows; value = 3*2*M*N*K FLOP / "
                   f"(quantize time + extrapolated GEMM time); OpenMP threads over rows = cores")}))


def reference_arm(args):
    rank, world, _ = _env_rank()
    if rank != 0:
        return None
    import torch
    cores = _host_cores()                      # the oracle's OpenMP rows and numpy's matmul use every core
    torch.set_num_threads(cores)
    import oracle
    oracle.build()
    m, n = args.ref_sample_m, args.ref_sample_n
    inputs = oracle_inputs(m, n, K)
    for _ in range(args.warmup):
        oracle_step(*inputs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(*inputs)
    dt = (time.perf_counter() - t0) / args.steps
    value = 3 * 2.0 * m * n * K / dt / 1e12
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle: FP32 steps emulated in FP64, FP64 GEMM)",
        "data": "synthetic", "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K,
                                        "sample": _oracle_sample_desc(m, n)},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": _oracle_sample_desc(m, n)},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def _time_ops(nv, ops, flush, stream, steps):
    """Total CUDA-event milliseconds of each op over `steps` passes (3
    untimed warm-up passes; L2 flushed by a write before every pass)."""
    import torch
    for _ in range(3):
        for _, fn in ops:
            fn()
    torch.cuda.synchronize()
    per = {name: 0.0 for name, _ in ops}
    evs = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in ops]
           for _ in range(steps)]
    for st in range(steps):
        flush.fill_(st & 0xFF)
        for (name, fn), (e0, e1) in zip(ops, evs[st]):
            e0.record(stream)
            fn()
            e1.record(stream)
    torch.cuda.synchronize()
    for st in range(steps):
        for (name, _), (e0, e1) in zip(ops, evs[st]):
            per[name] += e0.elapsed_time(e1)
    status = nv.nvfp4_sync_status()
    if status != nv.OK:
        raise RuntimeError(f"device status {status} after timing {[n for n, _ in ops]}")
    return per


def _time_steps(nv, step, flush, stream, steps):
    """Average CUDA-event milliseconds of `step` (3 untimed warm-up steps;
    L2 flushed by a write before every step, outside the events)."""
    import torch
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for st in range(steps):
        flush.fill_(st & 0xFF)
        evs[st][0].record(stream)
        step()
        evs[st][1].record(stream)
    torch.cuda.synchronize()
    status = nv.nvfp4_sync_status()
    if status != nv.OK:
        raise RuntimeError(f"device status {status} after timing a step")
    return sum(a.elapsed_time(b) for a, b in evs) / steps


def rht_rows_measure(nv, x, w, dy, flush, stream, steps):
    """Quantization of the Fprop and Dgrad operands with the 16-point RHT
    along their K (the transform the pages leave optional there): X and W
    rowwise RTN, dY rowwise SR, W^T colwise RTN.  Not part of `value`."""
    import workloads
    dev = x.device
    from quantize_block_scaled_amax_gb300 import empty_qtensor
    q = {name: empty_qtensor(r, c, dev) for name, (r, c) in
         dict(xq=(M, K), wq=(N, K), wtq=(K, N), dyq=(M, N)).items()}
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    ops = [
        ("rht_rows_x_rtn", lambda: nv.nvfp4_rht_quantize_rowwise(x, rht_seed=rh, out_rowwise=q["xq"])),
        ("rht_rows_w_rtn", lambda: nv.nvfp4_rht_quantize_rowwise(w, rht_seed=rh, out_rowwise=q["wq"])),
        ("rht_cols_w_rtn", lambda: nv.nvfp4_rht_quantize(w, rht_seed=rh, out_colwise=q["wtq"])),
        ("rht_rows_dy_sr", lambda: nv.nvfp4_rht_quantize_rowwise(dy, round="sr", seed=sr, rht_seed=rh,
                                                                 out_rowwise=q["dyq"])),
    ]
    bx, bw, bdy = M * K * 2, N * K * 2, M * N * 2
    nbytes = {"rht_rows_x_rtn": 2 * bx + M * K // 2 + M * K // 16, "rht_rows_w_rtn": 2 * bw + N * K // 2 + N * K // 16,
              "rht_cols_w_rtn": 2 * bw + N * K // 2 + N * K // 16,
              "rht_rows_dy_sr": 2 * bdy + M * N // 2 + M * N // 16}
    per = _time_ops(nv, ops, flush, stream, steps)
    return {name: {"ms": round(t / steps, 4), "gbs": round(nbytes[name] / (t / steps * 1e-3) / 1e9, 1)}
            for name, t in per.items()}


def bf16_gemm_measure(nv, x, w, flush, stream, steps, peaks):
    """The BF16 fallback GEMM (kind::f16) at the Fprop shape, for the layers
    the recipe keeps in high precision.  Not part of `value`."""
    import torch
    y = torch.empty(M, N, dtype=torch.bfloat16, device=x.device)
    per = _time_ops(nv, [("gemm_bf16_fprop", lambda: nv.nvfp4_gemm_bf16(x, w, out=y))], flush, stream, steps)
    ms = per["gemm_bf16_fprop"] / steps
    tf = 2.0 * M * N * K / (ms * 1e-3) / 1e12
    return {"ms": round(ms, 4), "tflops": round(tf, 1), "peak_bf16_tflops": peaks["bf16"],
            "frac": round(tf / peaks["bf16"], 4), "peak_source": f"{peaks['source']} cuBLAS bf16 burst"}


def ffn_measure(nv, flush, stream, steps, peaks, ms=(2048, 8192, 32768)):
    """The FFN block of the 12B model (up 5120 -> 20480, down 20480 -> 5120,
    no nonlinearity between them), forward and backward, at each token count:
    per step 6 GEMMs (Fprop, Dgrad, Wgrad of both linears) and the
    quantizations of the recipe, op by op through the C ABI as the main step.
    The down linear's input is the up linear's output and the up linear's
    output gradient is the down linear's input gradient.  Not part of `value`."""
    import torch
    import workloads
    from quantize_block_scaled_amax_gb300 import LinearContext
    d_model, d_ffn = workloads.D_MODEL, workloads.D_FFN
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    fp4_peak = peaks["bf16"] * FP4_OVER_BF16
    out = {}
    for m in ms:
        dev = flush.device
        x = workloads.activations(m, d_model, outliers=False, seed=workloads.SEED_BASE + 20, device=dev)
        w1 = workloads.weights(d_ffn, d_model, seed=workloads.SEED_BASE + 21, device=dev)
        w2 = workloads.weights(d_model, d_ffn, seed=workloads.SEED_BASE + 22, device=dev)
        dy2 = workloads.gradients(m, d_model, seed=workloads.SEED_BASE + 23, device=dev)
        c1, c2 = LinearContext(m, d_ffn, d_model, dev), LinearContext(m, d_model, d_ffn, dev)
        y1 = torch.empty(m, d_ffn, dtype=torch.bfloat16, device=dev)
        y2 = torch.empty(m, d_model, dtype=torch.bfloat16, device=dev)
        dy1 = torch.empty(m, d_ffn, dtype=torch.bfloat16, device=dev)      # = dX of the down linear
        dx = torch.empty(m, d_model, dtype=torch.bfloat16, device=dev)
        dw1 = torch.empty(d_ffn, d_model, dtype=torch.float32, device=dev)
        dw2 = torch.empty(d_model, d_ffn, dtype=torch.float32, device=dev)

        def lin(tag, c, xin, w, y):
            # X for Fprop and X^T (RHT) for Wgrad, one amax read (nvfp4_linear_fwd_rht)
            return [(f"{tag}_quant_x", lambda: nv.nvfp4_quantize_with_rht(xin, round="rtn", rht_seed=rh,
                                                                          out_rowwise=c.xq, out_colwise=c.xtq)),
                    (f"{tag}_quant_w", lambda: nv.nvfp4_quantize(w, block="16x16", colwise=True, out_rowwise=c.wq,
                                                                 out_colwise=c.wtq)),
                    (f"{tag}_gemm_fprop", lambda: nv.nvfp4_gemm(c.xq, c.wq, out=y))]

        def lin_bwd(tag, c, dyin, dxo, dwo):
            return [(f"{tag}_quant_dy", lambda: nv.nvfp4_quantize_with_rht(dyin, round="sr", seed=sr, rht_seed=rh,
                                                                           out_rowwise=c.dyq, out_colwise=c.dytq)),
                    (f"{tag}_gemm_dgrad", lambda: nv.nvfp4_gemm(c.dyq, c.wtq, out=dxo)),
                    (f"{tag}_gemm_wgrad", lambda: nv.nvfp4_gemm(c.dytq, c.xtq, out=dwo))]

        ops = (lin("up", c1, x, w1, y1) + lin("down", c2, y1, w2, y2) + lin_bwd("down", c2, dy2, dy1, dw2)
               + lin_bwd("up", c1, dy1, dx, dw1))

        def block_step():
            # the same step through the layer API (W quantized on the second stream)
            nv.nvfp4_linear_fwd(x, w1, c1, Y=y1, rht_seed=rh)
            nv.nvfp4_linear_fwd(y1, w2, c2, Y=y2, rht_seed=rh)
            nv.nvfp4_linear_bwd(dy2, None, c2, sr_seed=sr, rht_seed=rh, dX=dy1, dW=dw2)
            nv.nvfp4_linear_bwd(dy1, None, c1, sr_seed=sr, rht_seed=rh, dX=dx, dW=dw1)

        nsteps = max(3, steps if m <= 8192 else steps // 2)
        per = _time_ops(nv, ops, flush, stream, nsteps)
        ops_step_ms = sum(per.values()) / nsteps
        step_ms = _time_steps(nv, block_step, flush, stream, nsteps)
        flops = 6 * 2.0 * m * d_model * d_ffn
        gemm_ms = sum(v for k, v in per.items() if "gemm" in k) / nsteps
        quant_ms = ops_step_ms - gemm_ms
        # algorithmic bytes of the quantize ops: amax read + encode read + codes and scales per layout
        bx, bh = m * d_model, m * d_ffn
        # X of up and down, and dY of down and up: each rowwise + RHT colwise from one amax read
        qbytes = 2 * ((3 * 2 * bx + 2 * bx * 9 // 16) + (3 * 2 * bh + 2 * bh * 9 // 16))
        qbytes += 2 * (2 * 2 * d_model * d_ffn + 2 * d_model * d_ffn * 9 // 16)       # both W, 16x16 both layouts
        gemm_tf = 6 * 2.0 * m * d_model * d_ffn / (gemm_ms * 1e-3) / 1e12
        quant_gbs = qbytes / (quant_ms * 1e-3) / 1e9
        out[str(m)] = {"ms_per_step": round(step_ms, 4), "tflops": round(flops / (step_ms * 1e-3) / 1e12, 1),
                       "ms_per_step_ops": round(ops_step_ms, 4), "gemm_ms": round(gemm_ms, 4), "gemm_tflops": round(gemm_tf, 1),
                       "gemm_frac": round(gemm_tf / fp4_peak, 4), "quant_ms": round(quant_ms, 4),
                       "quant_gbs": round(quant_gbs, 1), "quant_frac": round(quant_gbs / peaks["hbm"], 4),
                       "steps": nsteps, "gpu_launches_per_step": 20, "gpu_launches_per_step_ops": 22,
                       "ops_ms": {k: round(v / nsteps, 4) for k, v in per.items()}}
        del x, w1, w2, dy2, c1, c2, y1, y2, dy1, dx, dw1, dw2, ops
        torch.cuda.empty_cache()
    return {"workload": "FFN block fwd+bwd of the 12B model (up 5120->20480, down 20480->5120), bf16 inputs, "
                        "6 NVFP4 GEMMs + the recipe's quantizations per step", "by_tokens": out,
            "peak_source": f"GEMM: {peaks['source']} burst bf16 x {FP4_OVER_BF16:g}; quantize: HBM copy"}


def mx_measure(nv, x, w, dy, flush, stream, steps):
    """The same layer step with MXFP4 operands (32-element blocks, UE8M0
    scales, no tensor scale: one read per quantize; weights 1x32 in both
    layouts, there being no 2D MXFP4 block), timed op by op like the main
    step.  Not part of `value`."""
    import torch
    import workloads
    dev = x.device
    q = {name: nv.empty_qtensor(r, c, dev, fmt="mxfp4") for name, (r, c) in
         dict(xq=(M, K), wq=(N, K), wtq=(K, N), dyq=(M, N), dytq=(N, M), xtq=(K, M)).items()}
    y = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
    dw = torch.empty(N, K, dtype=torch.float32, device=dev)
    sr, rh = workloads.SR_SEED, workloads.RHT_SEED
    ops = [
        ("quant_x_mx_rtn", lambda: nv.nvfp4_quantize(x, block="mx1x32", out_rowwise=q["xq"])),
        ("quant_w_mx_both", lambda: nv.nvfp4_quantize(w, block="mx1x32", colwise=True, out_rowwise=q["wq"],
                                                      out_colwise=q["wtq"])),
        ("gemm_fprop_mx", lambda: nv.nvfp4_gemm(q["xq"], q["wq"], out=y)),
        ("quant_dy_mx_sr", lambda: nv.nvfp4_quantize(dy, block="mx1x32", round="sr", seed=sr, out_rowwise=q["dyq"])),
        ("gemm_dgrad_mx", lambda: nv.nvfp4_gemm(q["dyq"], q["wtq"], out=dx)),
        ("rht_quant_dy_mx_sr", lambda: nv.nvfp4_rht_quantize(dy, round="sr", seed=sr, rht_seed=rh,
                                                             out_colwise=q["dytq"])),
        ("rht_quant_x_mx_rtn", lambda: nv.nvfp4_rht_quantize(x, rht_seed=rh, out_colwise=q["xtq"])),
        ("gemm_wgrad_mx", lambda: nv.nvfp4_gemm(q["dytq"], q["xtq"], out=dw)),
    ]
    # algorithmic bytes: one read of the input, codes, one UE8M0 byte per 32 elements per layout
    bx, bw, bdy = M * K * 2, N * K * 2, M * N * 2
    nbytes = {"quant_x_mx_rtn": bx + M * K // 2 + M * K // 32,
              "quant_w_mx_both": bw + 2 * (N * K // 2 + N * K // 32),
              "quant_dy_mx_sr": bdy + M * N // 2 + M * N // 32,
              "rht_quant_dy_mx_sr": bdy + M * N // 2 + M * N // 32,
              "rht_quant_x_mx_rtn": bx + M * K // 2 + M * K // 32}
    per = _time_ops(nv, ops, flush, stream, steps)
    out = {}
    for name, tot in per.items():
        ms = tot / steps
        if name.startswith("gemm"):
            out[name] = {"ms": round(ms, 4), "tflops": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1)}
        else:
            out[name] = {"ms": round(ms, 4), "gbs": round(nbytes[name] / (ms * 1e-3) / 1e9, 1)}
    step_ms = sum(per.values()) / steps
    return {"ms_per_step": round(step_ms, 4), "tflops": round(3 * 2.0 * M * N * K / (step_ms * 1e-3) / 1e12, 2),
            "steps": steps, "kernels": out,
            "note": "same layer step with MXFP4 operands (1x32 UE8M0 blocks, no tensor scale, no amax pass)"}


def profile_case(args):
    """One launch of one op of the step, for profiler captures: setup (input
    generation, quantization of the operands) runs first, then the op once."""
    import torch
    from quantize_block_scaled_amax_gb300 import build as _b
    _b.build()
    import quantize_block_scaled_amax_gb300 as nv
    import workloads
    m, n, k = args.m or M, args.n or N, args.k or K
    dev = torch.device("cuda", 0)
    op = args.profile
    if op == "gemm_pair":
        # the layer backward's Dgrad (dY 8192x20480 by W^T 5120x20480, bf16
        # out) and Wgrad (dY^T 20480x8192 by X^T 5120x8192, FP32 out) in one
        # launch, on operands of those shapes
        qs = []
        for r, c, seed in ((M, N, 31), (K, N, 32), (N, M, 33), (K, M, 34)):
            t = workloads.normal_with_outliers(r, c, p=0.001, factor=20.0, seed=workloads.SEED_BASE + seed,
                                               device=dev)
            qs.append(nv.nvfp4_quantize(t)[0])
            del t
        dx = torch.empty(M, K, dtype=torch.bfloat16, device=dev)
        dw = torch.empty(N, K, dtype=torch.float32, device=dev)
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        nv.nvfp4_gemm_pair(qs[0], qs[1], dx, qs[2], qs[3], dw)
    elif op.startswith("gemm"):
        x = workloads.activations(m, k, device=dev)
        w = workloads.weights(n, k, device=dev)
        qx, _ = nv.nvfp4_quantize(x)
        qw, _ = nv.nvfp4_quantize(w, block="16x16")
        del x, w
        torch.cuda.synchronize()
        torch.cuda.empty_cache()
        # "gemm_fp32": FP32 output, as the Wgrad GEMM writes it
        y = torch.empty(m, n, dtype=torch.float32 if op.endswith("fp32") else torch.bfloat16, device=dev)
        torch.cuda.synchronize()
        nv.nvfp4_gemm(qx, qw, out=y)
    elif op == "quant_x_rtn":
        x = workloads.activations(m, k, device=dev)
        torch.cuda.synchronize()
        nv.nvfp4_quantize(x)
    elif op == "quant_w_2d":
        w = workloads.weights(n, k, device=dev)
        torch.cuda.synchronize()
        nv.nvfp4_quantize(w, block="16x16", colwise=True)
    elif op == "quant_dy_sr":
        dy = workloads.gradients(m, n, device=dev)
        torch.cuda.synchronize()
        nv.nvfp4_quantize(dy, round="sr", seed=workloads.SR_SEED)
    elif op == "rht_x_rtn":
        # the RHT colwise RTN quantization of an activation (the FFN down
        # layer's input: 8192 x 20480 by default)
        x = workloads.activations(m, n, device=dev)
        torch.cuda.synchronize()
        nv.nvfp4_rht_quantize(x, rht_seed=workloads.RHT_SEED)
    elif op == "rht_dy_sr":
        dy = workloads.gradients(m, n, device=dev)
        torch.cuda.synchronize()
        nv.nvfp4_rht_quantize(dy, round="sr", seed=workloads.SR_SEED, rht_seed=workloads.RHT_SEED)
    else:
        raise SystemExit(f"unknown profile op {op}")
    torch.cuda.synchronize()
    st = nv.nvfp4_sync_status()
    if st != nv.OK:
        raise SystemExit(f"device status {st}")
    print(json.dumps({"profile": op, "m": m, "n": n, "k": k, "status": "ok"}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-mx", action="store_true",
                    help="skip the MXFP4 comparison step and the RHT-on-Fprop/Dgrad quantize timings")
    ap.add_argument("--no-ffn", action="store_true", help="skip the FFN block (up+down, M sweep) measurement")
    ap.add_argument("--cpu-baseline-only", default=None, choices=["full", "slice"])
    ap.add_argument("--cpu-sample-m", type=int, default=512)
    ap.add_argument("--cpu-sample-n", type=int, default=4096)
    ap.add_argument("--profile", default=None,
                    help="run one launch of one op: gemm_fprop, gemm, gemm_fp32, gemm_pair, quant_x_rtn, quant_w_2d, "
                         "quant_dy_sr, rht_dy_sr, rht_x_rtn")
    ap.add_argument("--m", type=int, default=0)
    ap.add_argument("--n", type=int, default=0)
    ap.add_argument("--k", type=int, default=0)
    ap.add_argument("--ref-sample-m", type=int, default=256)
    ap.add_argument("--ref-sample-n", type=int, default=1024)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.cpu_baseline_only:
        cpu_baseline_only(args.cpu_baseline_only, args.cpu_sample_m, args.cpu_sample_n)
        return
    if args.profile:
        profile_case(args)
        return
    out = reference_arm(args) if args.impl == "reference" else gpu_bench(args)
    if out is not None:
        print(json.dumps(out))


if __name__ == "__main__":
    main()
