"""Benchmark: routed-MoE decode on one DeepSeek-V4-Flash-shaped layer (hidden 4096, expert intermediate 2048,
256 routed experts, top-6, fp16 router), batch 1, 1000 independent seeded tokens, expert weights MXFP4
(also INT4 g32 and Q2_K with --fmt). One step = for each of the 1000 tokens: router top-6, then the fused
expert FFN (gate+up, SiLU*up, down, weighted combine), one token at a time, as a CUDA graph.

Prints one JSON line. value = tokens/s of the whole step; roofline = the fused FFN kernel's algorithmic bytes
(packed bytes of the token's 6 active experts) / its measured average launch time, against the measured HBM copy
bandwidth. The same run measures the other expert formats on the same weights and tokens (`formats`: INT4 g32,
Q2_K and MXFP4 in the mat-vec layout, each a router launch plus an FFN launch per token) and is the parity run:
the first 32 timed tokens' outputs (16 per extra format) are compared with the CPU oracle on the same seeds
(`parity`); a breach prints the line and exits with status 1. `--impl reference` times the CPU oracle on the host
cores instead (a bounded sample of the workload).
"""
from __future__ import annotations

import argparse
import concurrent.futures as cf
import json
import os
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

H, I, E, K_TOP, NTOK = 4096, 2048, 256, 6, 1000
FMT_IDS = {"mxfp4": 1, "int4g32": 2, "q2k": 3}


def max_over_ranks(value: float, dist, device) -> float:
    """The largest of the ranks' values (a timed region lasts as long as its slowest replica); `value` itself
    with one process (dist None)."""
    if dist is None:
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def rank_token_seed(seed: int, rank: int) -> int:
    """Seed of the tokens a replica decodes: every rank decodes tokens of its own."""
    return seed + rank * 7919


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=5)
    p.add_argument("--warmup", type=int, default=3)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--fmt", default="mxfp4", choices=list(FMT_IDS))
    p.add_argument("--tokens", type=int, default=NTOK)
    p.add_argument("--seed", type=int, default=1)
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-verify", action="store_true", help="skip the verify-cost and speculative-acceptance measurements")
    p.add_argument("--cpu-seconds", type=float, default=15.0)
    p.add_argument("--experts", type=int, default=E, help="expert slots of the layer (smaller only for profiling)")
    p.add_argument("--layout", default="auto", choices=["auto", "tc", "decode"],
                   help="weight layout of the decode path: tc (MXFP4, tcgen05 kernels) or decode (mat-vec kernels); "
                        "auto = tc for MXFP4, decode otherwise")
    p.add_argument("--no-formats", action="store_true", help="measure only the --fmt / --layout path")
    p.add_argument("--no-stack", action="store_true", help="skip the 43-layer stack measurement")
    p.add_argument("--no-shared", action="store_true", help="skip the routed + Q8_0 shared-expert measurement")
    p.add_argument("--stack-tokens", type=int, default=64, help="tokens per timed pass of the 43-layer stack")
    p.add_argument("--no-parity", action="store_true", help="skip the oracle comparison of the timed tokens")
    p.add_argument("--parity-tokens", type=int, default=32)
    p.add_argument("--prefill-tokens", type=int, default=4096,
                   help="tokens of the prefill grouped-GEMM measurement (MXFP4 only; 0 = skip)")
    return p.parse_args()


def measured_peaks():
    try:
        return json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json")))
    except Exception:
        return None


def peak_of(peaks, key: str):
    """One measured peak from MEASURED_PEAKS.json: a positive number stored under `key` directly or as
    {"value": number}; None when the file, the key or a usable number is missing (the caller then falls back)."""
    if not isinstance(peaks, dict):
        return None
    v = peaks.get(key)
    if isinstance(v, dict):
        v = v.get("value")
    try:
        v = float(v)
    except (TypeError, ValueError):
        return None
    return v if v > 0 else None


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 200 ms while the timed region runs."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 7:
                continue
            try:
                sm.append(float(f[0]))
                mx = float(f[1])
            except ValueError:
                continue
            for n, v in zip(names, f[3:7]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": mx, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------ GPU arm
def run_ours(args):
    import torch
    import bit_moe_decode_gb300 as m
    from moe_inputs import GATE, UP, DOWN, expert_stack_f32, router_f16_bits, x_bf16_bits

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dist = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    if m.moe_check_device() != 0:
        raise RuntimeError("libmoe: device is not sm_103")
    fmt = FMT_IDS[args.fmt]
    T = args.tokens
    E = args.experts
    do_prefill = args.prefill_tokens > 0 and fmt == 1
    use_tc = fmt == 1 and args.layout != "decode"

    # ---- weights: seeded fp32 -> packed on the GPU by the library's encoder (replica per rank, same weights)
    layer_tc = m.Layer(fmt, H, I, E, layout=m.MOE_LAYOUT_TC, device=dev) if (use_tc or do_prefill) else None
    layer = layer_tc if use_tc else m.Layer(fmt, H, I, E, device=dev)
    layer_p = layer_tc if do_prefill else None
    # the other formats, measured on the same weights and tokens (single GPU only: the scaling runs time the headline)
    extra = {}
    if not args.no_formats and world == 1:
        for name, fid in FMT_IDS.items():
            if name == args.fmt and not use_tc:
                continue
            extra[name if name != "mxfp4" else "mxfp4_matvec_layout"] = m.Layer(fid, H, I, E, device=dev)
    t0 = time.time()
    batch = 16
    pool = cf.ThreadPoolExecutor(2)

    def gen(e0):
        ex = range(e0, min(E, e0 + batch))
        return [expert_stack_f32(args.seed, 0, ex, which, H, I) for which in (GATE, UP, DOWN)]

    fut = pool.submit(gen, 0)
    for e0 in range(0, E, batch):
        g, u, d = fut.result()
        if e0 + batch < E:
            fut = pool.submit(gen, e0 + batch)
        gd, ud, dd = torch.from_numpy(g).to(dev), torch.from_numpy(u).to(dev), torch.from_numpy(d).to(dev)
        layer.pack(m.MOE_SRC_F32, gd, ud, dd, e0=e0)
        if layer_tc is not None and layer_tc is not layer:
            layer_tc.pack(m.MOE_SRC_F32, gd, ud, dd, e0=e0)
        for lx in extra.values():
            lx.pack(m.MOE_SRC_F32, gd, ud, dd, e0=e0)
    torch.cuda.synchronize()
    setup_s = time.time() - t0

    wr = torch.from_numpy(router_f16_bits(args.seed, 0, E, H).view(np.int16)).to(dev)
    x_host = x_bf16_bits(rank_token_seed(args.seed, rank), range(T), H)   # each rank decodes its own tokens
    x = torch.from_numpy(x_host.view(np.int16)).to(dev)
    idx = torch.zeros((T, K_TOP), dtype=torch.int32, device=dev)
    w = torch.zeros((T, K_TOP), dtype=torch.float32, device=dev)
    y = torch.zeros((T, H), dtype=torch.float32, device=dev)
    ws = layer.workspace(1, K_TOP)
    stream = torch.cuda.Stream(device=dev)

    fused = use_tc and E <= 256   # router + FFN in one launch (the router's logits spread over the whole grid)

    def step_launch():
        for t in range(T):
            if fused:
                m.moe_route_expert_ffn(layer, wr, x[t], 1, K_TOP, idx[t], w[t], y[t], None, False, ws, stream=stream)
            else:
                m.moe_route_topk(wr, x[t], 1, H, E, K_TOP, None, None, 0, idx[t], w[t], stream=stream)
                m.moe_expert_ffn_decode(layer, x[t], idx[t], w[t], K_TOP, y[t], None, False, ws, stream=stream)

    def ffn_only_launch():
        for t in range(T):
            m.moe_expert_ffn_decode(layer, x[t], idx[t], w[t], K_TOP, y[t], None, False, ws, stream=stream)

    idx2 = torch.zeros_like(idx)
    w2 = torch.zeros_like(w)

    def route_only_launch():
        for t in range(T):
            m.moe_route_topk(wr, x[t], 1, H, E, K_TOP, None, None, 0, idx2[t], w2[t], stream=stream)

    with torch.cuda.stream(stream):
        step_launch()   # warm the attribute setup outside capture
    stream.synchronize()
    if m.moe_get_device_status(ws, stream) != 0:
        raise RuntimeError("device status after warm-up")
    use_graph = True
    try:
        g_step = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_step, stream=stream):
            step_launch()
        g_ffn = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_ffn, stream=stream):
            ffn_only_launch()
        g_route = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_route, stream=stream):
            route_only_launch()
    except Exception as ex:  # capture unsupported: launch eagerly (host launch cost then counts)
        print("graph capture failed (%s); timing eager launches" % ex, file=sys.stderr)
        use_graph = False

    def run_step():
        with torch.cuda.stream(stream):
            if use_graph:
                g_step.replay()
            else:
                step_launch()

    def run_ffn():
        with torch.cuda.stream(stream):
            if use_graph:
                g_ffn.replay()
            else:
                ffn_only_launch()

    for _ in range(args.warmup):
        run_step()
    stream.synchronize()

    # ---- timed region: K steps, barrier + sync on both sides, events on the launching stream
    if dist:
        dist.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for _ in range(args.steps):
        run_step()
    ev1.record(stream)
    ev1.synchronize()
    torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    clk = clocks.stop()
    if dist:
        ms = max_over_ranks(ms, dist, dev)
        dist.barrier()
    status = m.moe_get_device_status(ws, stream)
    if status != 0:
        raise RuntimeError("device status %d after timed region" % status)
    npar = 0 if args.no_parity else min(args.parity_tokens, T)
    checks = []
    if npar and rank == 0:   # the timed step's own outputs (every step computes the same y)
        checks.append((None, fmt, y[:npar].cpu().numpy(), idx[:npar].cpu().numpy(), w[:npar].cpu().numpy()))

    # ---- the dominant kernel alone (routing fixed): average launch duration
    for _ in range(2):
        run_ffn()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    reps = max(2, args.steps)
    for _ in range(reps):
        run_ffn()
    e1.record(stream)
    e1.synchronize()
    ffn_us = e0.elapsed_time(e1) * 1e3 / (reps * T)
    route_us = None
    if use_graph:
        with torch.cuda.stream(stream):
            g_route.replay()
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g_route.replay()
        e1.record(stream)
        e1.synchronize()
        route_us = e0.elapsed_time(e1) * 1e3 / (reps * T)
        assert torch.equal(idx2, idx), "router results differ between runs"
    # routing alone
    idx_np = idx.cpu().numpy()
    uniq = np.mean([len(set(r)) for r in idx_np])
    lay = 1 if use_tc else 0
    per_expert = m.moe_packed_bytes(fmt, lay, 0, 1, H, I) + m.moe_packed_bytes(fmt, lay, 1, 1, H, I)
    alg_bytes = float(np.mean([len(set(r)) for r in idx_np])) * per_expert

    # ---- end to end through the public API with host buffers (pinned), copies inside the timed region
    xh = torch.from_numpy(x_host.view(np.int16)).pin_memory()
    yh = torch.empty((T, H), dtype=torch.float32).pin_memory()
    torch.cuda.synchronize()
    e2e_steps = max(1, min(args.steps, 3))
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s0.record(stream)
    for _ in range(e2e_steps):
        with torch.cuda.stream(stream):
            x.copy_(xh, non_blocking=True)
        run_step()
        with torch.cuda.stream(stream):
            yh.copy_(y, non_blocking=True)
    s1.record(stream)
    s1.synchronize()
    e2e_ms = s0.elapsed_time(s1) / e2e_steps
    e2e_ms = max_over_ranks(e2e_ms, dist, dev)

    formats = {}
    for key, lx in extra.items():
        formats[key], rows = bench_format(m, torch, args, dev, stream, lx, wr, x, x_host, min(npar, 16))
        if rows is not None:
            checks.append((key, lx.fmt) + rows)
    shared = None
    if fused and world == 1 and not args.no_shared:
        shared, rows = bench_shared(m, torch, args, dev, stream, layer, wr, x, x_host, min(npar, 8))
        if rows is not None:
            checks.append(("shared_expert", None) + rows)
    prefill = bench_prefill(m, torch, args, dev, stream, layer_p, E) if do_prefill else None
    stack = None
    if not args.no_stack and world == 1 and fmt == 1:
        stack = bench_stack(m, torch, args, dev, stream)
    verify = bench_verify(m, torch, args, dev, stream, layer, wr, x_host, E, per_expert) if (use_tc and not args.no_verify) else None
    spec = bench_spec(m, torch, dev, stream) if not args.no_verify else None

    out = None
    if rank == 0:
        hbm_measured = peak_of(measured_peaks(), "hbm_gbs")
        peak = hbm_measured or 6800.0
        achieved = alg_bytes / (ffn_us * 1e-6) / 1e9
        ms_step = ms / args.steps
        value = world * T / (ms_step * 1e-3)
        out = {
            "metric": "routed-MoE decode tok/s and HBM GB/s (% of 8 TB/s), MXFP4/Q2_K/INT4 experts",
            "value": round(value, 1), "unit": "tok/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_step, 4), "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": {1: "mxfp4", 2: "int4g32", 3: "q2k"}[fmt] + " weights, bf16 x, " +
                     ("E2M1-part activations (6 parts), block-scaled tcgen05 kind::mxf4, fp32 accumulate" if use_tc else "fp16/fp32 mma"),
            "data": "synthetic (seeded N(0,0.02) weights quantised on the GPU, N(0,1) bf16 tokens)",
            "config": {"workload": "DS4-Flash routed-MoE layer decode, batch 1, %d independent tokens" % T,
                       "H": H, "I": I, "experts": E, "top_k": K_TOP, "format": args.fmt,
                       "layout": "tc" if use_tc else "decode",
                       "l2": "inputs larger than L2 (3.4 GB of experts, random routing)",
                       "parallelism": "replicas" if world > 1 else "single GPU"},
            "gpu_launches": (1 if fused else 2) * T * args.steps,
            "step_kernels": "moe_route_expert_ffn (router + FFN, one launch)" if fused else "moe_route_topk + moe_expert_ffn_decode",
            "hbm_gbs_step": round(alg_bytes * T / (ms_step * 1e-3) / 1e9, 1),
            "pct_of_8tbs_step": round(100 * alg_bytes * T / (ms_step * 1e-3) / 8e12, 2),
            "ffn_kernel_us": round(ffn_us, 3),
            "route_kernel_us": round(route_us, 3) if route_us else None,
            "ffn_tok_s": round(1e6 / ffn_us, 1),
            "ffn_pct_of_8tbs": round(100 * alg_bytes / (ffn_us * 1e-6) / 8e12, 2),
            "mean_unique_experts": float(uniq),
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4),
                         # DRAM bytes per launch come from an ncu capture of the kernel, not from this run
                         "traffic": None,
                         "kernel": "decode_kernel (tcgen05)" if use_tc else "ffn_kernel<%s>" % args.fmt,
                         "bytes_per_launch": alg_bytes,
                         "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if hbm_measured else "fallback"},
            "e2e": {"value": round(world * T / (e2e_ms * 1e-3), 1), "unit": "tok/s",
                    "h2d_bytes_per_step": int(T * H * 2), "d2h_bytes_per_step": int(T * H * 4)},
            "clocks": clk,
            "formats": formats,
            "shared_expert": shared,
            "stack": stack,
            "prefill": prefill,
            "verify": verify,
            "spec_accept": spec,
            "setup_s": round(setup_s, 1),
            "cuda_graph": use_graph,
        }
    if dist:
        dist.destroy_process_group()
    return out, checks


def bench_format(m, torch, args, dev, stream, layer, wr, x, x_host, npar):
    """One more expert format on the same weights and tokens, in the mat-vec (DECODE) layout: a step is, per token,
    the router launch (moe_route_topk) and the FFN launch (moe_expert_ffn_decode), replayed as a CUDA graph. Reports
    the step, the FFN launch alone (routing fixed) against the HBM roofline, and the step end to end with host
    buffers; returns the first npar tokens' (y, idx, w) for the oracle comparison."""
    T = x.shape[0]
    fid = layer.fmt
    ws = layer.workspace(1, K_TOP)
    idx = torch.zeros((T, K_TOP), dtype=torch.int32, device=dev)
    w = torch.zeros((T, K_TOP), dtype=torch.float32, device=dev)
    y = torch.zeros((T, H), dtype=torch.float32, device=dev)

    def step_launch():
        for t in range(T):
            m.moe_route_topk(wr, x[t], 1, H, layer.E, K_TOP, None, None, 0, idx[t], w[t], stream=stream)
            m.moe_expert_ffn_decode(layer, x[t], idx[t], w[t], K_TOP, y[t], None, False, ws, stream=stream)

    def ffn_launch():
        for t in range(T):
            m.moe_expert_ffn_decode(layer, x[t], idx[t], w[t], K_TOP, y[t], None, False, ws, stream=stream)

    with torch.cuda.stream(stream):
        step_launch()
    stream.synchronize()
    if m.moe_get_device_status(ws, stream) != 0:
        raise RuntimeError("device status after the warm-up of format %d" % fid)
    g_step, g_ffn = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        step_launch()
    with torch.cuda.graph(g_ffn, stream=stream):
        ffn_launch()

    def timed(g, reps):
        with torch.cuda.stream(stream):
            for _ in range(max(1, args.warmup)):
                g.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                g.replay()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    reps = max(1, args.steps)
    ms_step = timed(g_step, reps)
    ffn_us = timed(g_ffn, reps) * 1e3 / T
    # end to end: the tokens from pinned host memory and the outputs back, inside the timed region
    xh = torch.from_numpy(x_host.view(np.int16)).pin_memory()
    yh = torch.empty((T, H), dtype=torch.float32).pin_memory()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_e2e = max(1, min(reps, 3))
    e0.record(stream)
    for _ in range(n_e2e):
        with torch.cuda.stream(stream):
            x.copy_(xh, non_blocking=True)
            g_step.replay()
            yh.copy_(y, non_blocking=True)
    e1.record(stream)
    e1.synchronize()
    e2e_ms = e0.elapsed_time(e1) / n_e2e
    if m.moe_get_device_status(ws, stream) != 0:
        raise RuntimeError("device status after format %d" % fid)
    idx_np = idx.cpu().numpy()
    per_expert = m.moe_packed_bytes(fid, 0, 0, 1, H, I) + m.moe_packed_bytes(fid, 0, 1, 1, H, I)
    alg = float(np.mean([len(set(r)) for r in idx_np])) * per_expert
    peak = peak_of(measured_peaks(), "hbm_gbs")
    achieved = alg / (ffn_us * 1e-6) / 1e9
    res = {"layout": "matvec (DECODE)", "kernel": "ffn_kernel<%s>" % {1: "mxfp4", 2: "int4g32", 3: "q2k"}[fid],
           "step_kernels": "moe_route_topk + moe_expert_ffn_decode",
           "tok_s": round(T / (ms_step * 1e-3), 1), "ms_per_step": round(ms_step, 4),
           "ffn_kernel_us": round(ffn_us, 3), "gpu_launches": 2 * T * reps,
           "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak or 6800.0, "unit": "GB/s",
                        "frac": round(achieved / (peak or 6800.0), 4), "traffic": None, "bytes_per_launch": alg,
                        "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peak else "fallback"},
           "e2e": {"value": round(T / (e2e_ms * 1e-3), 1), "unit": "tok/s", "h2d_bytes_per_step": int(T * H * 2),
                   "d2h_bytes_per_step": int(T * H * 4)}}
    rows = (y[:npar].cpu().numpy(), idx[:npar].cpu().numpy(), w[:npar].cpu().numpy()) if npar else None
    return res, rows


N_SHARED = 8   # shared-expert copies the tokens rotate over (8 x 26.7 MB > L2), standing in for 8 layers' own


def bench_shared(m, torch, args, dev, stream, layer, wr, x, x_host, npar):
    """The routed layer plus the always-on shared expert in Q8_0 (hidden 4096, intermediate 2048): per token the
    fused router + routed FFN launch writes y, then the shared expert runs as a one-expert Q8_0 layer
    (moe_expert_ffn_decode, idx 0 of its own layer, w 1, accumulate) and writes the bf16 copy. Token t reads shared
    expert t % 8, so that the shared weights come from HBM as they do when every layer has its own. Reports the
    combined step and the shared launch alone against the HBM roofline; returns the first npar tokens' rows for the
    oracle comparison."""
    from moe_inputs import GATE, UP, DOWN, expert_stack_f32
    T = x.shape[0]
    sh = m.Layer(4, H, I, N_SHARED, device=dev)
    g, u, d = (torch.from_numpy(expert_stack_f32(args.seed, 1, range(N_SHARED), which, H, I)).to(dev)
               for which in (GATE, UP, DOWN))
    sh.pack(m.MOE_SRC_F32, g, u, d)
    del g, u, d
    ws_r, ws_s = layer.workspace(1, K_TOP), sh.workspace(1, 1)
    idx = torch.zeros((T, K_TOP), dtype=torch.int32, device=dev)
    w = torch.zeros((T, K_TOP), dtype=torch.float32, device=dev)
    y = torch.zeros((T, H), dtype=torch.float32, device=dev)
    yb = torch.zeros((T, H), dtype=torch.int16, device=dev)
    sidx = (torch.arange(T, dtype=torch.int32, device=dev) % N_SHARED).reshape(T, 1).contiguous()
    sw = torch.ones((T, 1), dtype=torch.float32, device=dev)

    def step_launch():
        for t in range(T):
            m.moe_route_expert_ffn(layer, wr, x[t], 1, K_TOP, idx[t], w[t], y[t], None, False, ws_r, stream=stream)
            m.moe_expert_ffn_decode(sh, x[t], sidx[t], sw[t], 1, y[t], yb[t], True, ws_s, stream=stream)

    def shared_launch():
        for t in range(T):
            m.moe_expert_ffn_decode(sh, x[t], sidx[t], sw[t], 1, y[t], yb[t], True, ws_s, stream=stream)

    with torch.cuda.stream(stream):
        step_launch()
    stream.synchronize()
    if m.moe_get_device_status(ws_r, stream) != 0 or m.moe_get_device_status(ws_s, stream) != 0:
        raise RuntimeError("device status after the shared-expert warm-up")
    g_step, g_sh = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
    with torch.cuda.graph(g_step, stream=stream):
        step_launch()
    with torch.cuda.graph(g_sh, stream=stream):
        shared_launch()

    def timed(gr, reps):
        with torch.cuda.stream(stream):
            for _ in range(max(1, args.warmup)):
                gr.replay()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(reps):
                gr.replay()
        e1.record(stream)
        e1.synchronize()
        return e0.elapsed_time(e1) / reps

    reps = max(1, args.steps)
    sh_us = timed(g_sh, reps) * 1e3 / T
    ms_step = timed(g_step, reps)   # last: y holds one step's routed + shared output
    if m.moe_get_device_status(ws_r, stream) != 0 or m.moe_get_device_status(ws_s, stream) != 0:
        raise RuntimeError("device status after the shared-expert measurement")
    alg = m.moe_packed_bytes(4, 0, 0, 1, H, I) + m.moe_packed_bytes(4, 0, 1, 1, H, I)
    peak = peak_of(measured_peaks(), "hbm_gbs")
    achieved = alg / (sh_us * 1e-6) / 1e9
    res = {"format": "q8_0 (34 B per 32 weights)", "shared_experts": N_SHARED,
           "step_kernels": "moe_route_expert_ffn (routed) + moe_expert_ffn_decode (shared, Q8_0, accumulate)",
           "tok_s": round(T / (ms_step * 1e-3), 1), "us_per_token": round(ms_step * 1e3 / T, 3),
           "shared_kernel_us": round(sh_us, 3), "gpu_launches": 2 * T * reps,
           "roofline_shared": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak or 6800.0, "unit": "GB/s",
                               "frac": round(achieved / (peak or 6800.0), 4), "traffic": None,
                               "kernel": "ffn_kernel<q8_0>", "bytes_per_launch": alg,
                               "peak_source": "MEASURED_PEAKS.json hbm_gbs (of measured)" if peak else "fallback"}}
    rows = None
    if npar:
        rows = (y[:npar].cpu().numpy(), idx[:npar].cpu().numpy(), w[:npar].cpu().numpy(),
                sidx[:npar, 0].cpu().numpy(), yb[:npar].cpu().numpy().view(np.uint16))
    return res, rows


def bench_stack(m, torch, args, dev, stream, n_layers=43, n_hash=3, vocab=32768):
    """The whole routed-expert stack: 43 layers x 256 MXFP4 experts in the tensor-core layout (147 GB, generated on
    the GPU: seeded N(0, 0.02) fp32 per expert, packed by the library's encoder), layers 0-2 routed by a seeded
    tid2eid table (vocab 32768, 6 distinct experts, w = 1/6), layers 3-42 by their own fp16 router (fused into the
    FFN launch); layer L + 1's x = bf16(y_L / rms(y_L)) (moe_rms_norm_bf16: the model normalises before each MoE
    layer, and an unnormalised chain of random layers collapses to zero, where routing degenerates to ties). Each
    layer also holds a Q8_0 shared expert (intermediate 2048), timed
    separately (`with_shared_experts`: decode and T = 8 verify with the shared expert after every routed call). Decode: args.stack_tokens tokens one at a time, all layers, as a CUDA
    graph; verify: the same tokens in batches of T = 2, 4, 8 (independent routing: each layer sweeps the union of
    the batch's experts). Algorithmic bytes = packed bytes of each layer's union of experts, summed over layers."""
    from bit_moe_decode_gb300.stack import RoutedStack
    from moe_inputs import tid2eid, token_ids, x_bf16_bits
    per_expert = m.moe_packed_bytes(1, 1, 0, 1, H, I) + m.moe_packed_bytes(1, 1, 1, 1, H, I)
    per_shared = m.moe_packed_bytes(4, 0, 0, 1, H, I) + m.moe_packed_bytes(4, 0, 1, 1, H, I)   # Q8_0, intermediate I
    need = n_layers * (E * per_expert + per_shared)
    free, _ = torch.cuda.mem_get_info(dev)
    if free < need + (8 << 30):
        return {"skipped": "needs %.1f GB of free device memory, %.1f GB free" % (need / 1e9, free / 1e9)}
    t0 = time.time()
    st = RoutedStack(H, I, E, K_TOP, n_layers, n_hash, vocab, T_max=8, device=dev, shared_I=I)
    gen = torch.Generator(device=dev)
    batch = 32
    for L in range(n_layers):
        gen.manual_seed(args.seed * 1000 + L)
        for e0 in range(0, E, batch):
            g = torch.randn((batch, I, H), generator=gen, device=dev).mul_(0.02)
            u = torch.randn((batch, I, H), generator=gen, device=dev).mul_(0.02)
            d = torch.randn((batch, H, I), generator=gen, device=dev).mul_(0.02)
            st.layers[L].pack(m.MOE_SRC_F32, g, u, d, e0=e0, stream=torch.cuda.current_stream(dev))
        if L < n_hash:
            st.tid2eid[L] = torch.from_numpy(tid2eid(args.seed, L, vocab, E, K_TOP)).to(dev)
        else:
            st.router[L] = (torch.randn((E, H), generator=gen, device=dev) * 0.02).half().view(torch.int16)
        gen.manual_seed(args.seed * 1000 + 500 + L)   # the layer's shared expert, from a stream of its own
        g = torch.randn((1, I, H), generator=gen, device=dev).mul_(0.02)
        u = torch.randn((1, I, H), generator=gen, device=dev).mul_(0.02)
        d = torch.randn((1, H, I), generator=gen, device=dev).mul_(0.02)
        st.shared[L].pack(m.MOE_SRC_F32, g, u, d, stream=torch.cuda.current_stream(dev))
    del g, u, d
    torch.cuda.synchronize()
    setup_s = time.time() - t0
    N = max(8, (args.stack_tokens // 8) * 8)
    toks = torch.from_numpy(token_ids(args.seed, N, vocab)).to(dev)
    xs = torch.from_numpy(x_bf16_bits(args.seed + 31, range(N), H).view(np.int16)).to(dev)

    res, unions, res_sh = {}, {}, {}
    for T, sh in ((1, False), (2, False), (4, False), (8, False), (1, True), (8, True)):
        def launch(T=T, sh=sh):
            for j in range(N // T):
                st.run(T, token_ids=toks[j * T:(j + 1) * T], x0=xs[j * T:(j + 1) * T], stream=stream, shared=sh)
        # the routing of every pass (eager, once): each layer's union of experts over the batch
        us = []
        for j in range(N // T):
            with torch.cuda.stream(stream):
                st.run(T, token_ids=toks[j * T:(j + 1) * T], x0=xs[j * T:(j + 1) * T], stream=stream, shared=sh)
            stream.synchronize()
            us.append([len(np.unique(st.idx[L][:T].cpu().numpy())) for L in range(n_layers)])
        if not sh:
            unions[T] = float(np.mean(np.sum(us, axis=1)))   # union sizes summed over the layers, per pass
        s1, s2 = m.moe_get_device_status(st.ws, stream), m.moe_get_device_status(st.ws_shared, stream)
        if s1 != 0 or s2 != 0:
            raise RuntimeError("device status after the stack's eager pass (T = %d, shared = %d): routed %d, shared %d"
                               % (T, sh, s1, s2))
        g_ = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_, stream=stream):
            launch()
        times = []
        for _ in range(max(1, args.warmup)):
            with torch.cuda.stream(stream):
                g_.replay()
        for _ in range(3):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                g_.replay()
            e1.record(stream)
            e1.synchronize()
            times.append(e0.elapsed_time(e1))
        (res_sh if sh else res)[T] = float(np.median(times)) / (N // T)   # ms per pass of T tokens
        s1, s2 = m.moe_get_device_status(st.ws, stream), m.moe_get_device_status(st.ws_shared, stream)
        if s1 != 0 or s2 != 0:
            raise RuntimeError("device status after the stack (T = %d, shared = %d): routed %d, shared %d"
                               % (T, sh, s1, s2))
    peak = peak_of(measured_peaks(), "hbm_gbs") or 6800.0
    t1 = res[1]
    bytes1 = unions[1] * per_expert
    # each layer's Q8_0 shared expert (intermediate I) after its routed call: one more launch per layer
    ts1, bs1 = res_sh[1], bytes1 + n_layers * per_shared
    shared_line = {"decode": {"tok_s": round(1e3 / ts1, 2), "us_per_token": round(ts1 * 1e3, 2),
                              "bytes_per_token": bs1, "gbs": round(bs1 / (ts1 * 1e-3) / 1e9, 1),
                              "frac": round(bs1 / (ts1 * 1e-3) / 1e9 / peak, 4),
                              "gpu_launches_per_token": st.launches_per_run(shared=True)},
                   "verify_T8": {"us_per_pass": round(res_sh[8] * 1e3, 2), "raw_ratio": round(res_sh[8] / ts1, 3)},
                   "shared_bytes_per_layer": per_shared}
    out = {"workload": "%d layers x %d MXFP4 experts (%.1f GB resident, generated on the GPU), layers 0-%d hash-routed "
                       "(tid2eid, vocab %d), the rest softmax top-%d (router fused), layer L+1's x = bf16(rmsnorm(y_L)); %d "
                       "tokens per timed pass" % (n_layers, E, st.packed_bytes() / 1e9, n_hash - 1, vocab, K_TOP, N),
           "decode": {"tok_s": round(1e3 / t1, 2), "us_per_token": round(t1 * 1e3, 2),
                      "bytes_per_token": bytes1, "gbs": round(bytes1 / (t1 * 1e-3) / 1e9, 1),
                      "roofline": {"bound": "hbm", "achieved": round(bytes1 / (t1 * 1e-3) / 1e9, 1), "peak": peak,
                                   "unit": "GB/s", "frac": round(bytes1 / (t1 * 1e-3) / 1e9 / peak, 4),
                                   "traffic": None},
                      "gpu_launches_per_token": st.launches_per_run()},
           "verify": {"us_per_pass": {str(T): round(res[T] * 1e3, 2) for T in res},
                      "tok_s": {str(T): round(T * 1e3 / res[T], 2) for T in res},
                      "union_experts_over_layers": {str(T): round(unions[T], 1) for T in res},
                      "raw_ratio": {str(T): round(res[T] / t1, 3) for T in res},
                      "per_union_byte_ratio": {str(T): round(res[T] / (t1 * unions[T] / unions[1]), 3) for T in res}},
           "with_shared_experts": shared_line,
           "setup_s": round(setup_s, 1)}
    del st
    torch.cuda.empty_cache()
    return out


def bench_verify(m, torch, args, dev, stream, layer, wr, x_host, E, per_expert):
    """Verify cost (speculative verify of T = 1, 2, 4, 8 tokens in one sweep) on the same layer:
    (i) shared routing: the T tokens all use the first token's experts, t(8) / t(1);
    (ii) independent routing: t(T) / (t(1) * U_T / 6), U_T = union of the tokens' experts;
    (iii) raw t(T) / t(1). Each t is the mean over 200 calls of a CUDA graph (the window of tokens advances)."""
    n_calls = 200
    xs = torch.from_numpy(x_host.view(np.int16)).to(dev)
    nt = xs.shape[0]
    ws = layer.workspace(8, K_TOP)
    idx_all = torch.zeros((nt, K_TOP), dtype=torch.int32, device=dev)
    w_all = torch.zeros((nt, K_TOP), dtype=torch.float32, device=dev)
    m.moe_route_topk(wr, xs, nt, H, E, K_TOP, None, None, 0, idx_all, w_all, stream=stream)
    stream.synchronize()
    idx_np = idx_all.cpu().numpy()
    out = {}
    y = torch.zeros((8, H), dtype=torch.float32, device=dev)
    for shared in (False, True):
        res = {}
        for T in (1, 2, 4, 8):
            starts = [(i * T) % (nt - 8) for i in range(n_calls)]
            if shared:   # every token of the window routed (and weighted) like the window's first token
                sidx = torch.stack([idx_all[st].expand(T, -1) for st in starts]).contiguous()
                sw = torch.stack([w_all[st].expand(T, -1) for st in starts]).contiguous()
                args_of = [(xs[st:st + T], sidx[i], sw[i]) for i, st in enumerate(starts)]
                u = float(np.mean([len(set(idx_np[st])) for st in starts]))
            else:
                args_of = [(xs[st:st + T], idx_all[st:st + T], w_all[st:st + T]) for st in starts]
                u = float(np.mean([len(set(idx_np[st:st + T].ravel())) for st in starts]))

            def launch():
                for xa, ia, wa in args_of:
                    m.moe_expert_ffn_verify(layer, xa, T, ia, wa, K_TOP, y, None, False, ws, stream=stream)
            with torch.cuda.stream(stream):
                launch()
            stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                launch()
            with torch.cuda.stream(stream):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            with torch.cuda.stream(stream):
                g.replay()
                g.replay()
            e1.record(stream)
            e1.synchronize()
            res[T] = (e0.elapsed_time(e1) * 1e3 / (2 * n_calls), u)
        t1, u1 = res[1]
        key = "shared_routing" if shared else "independent_routing"
        out[key] = {"us": {str(T): round(res[T][0], 3) for T in res},
                    "union_experts": {str(T): round(res[T][1], 2) for T in res},
                    "raw_ratio": {str(T): round(res[T][0] / t1, 3) for T in res},
                    "per_union_byte_ratio": {str(T): round(res[T][0] / (t1 * res[T][1] / u1), 3) for T in res},
                    "gbs": {str(T): round(res[T][1] * per_expert / (res[T][0] * 1e-6) / 1e9, 1) for T in res}}
    if m.moe_get_device_status(ws, stream) != 0:
        raise RuntimeError("device status after the verify measurements")
    return out


def bench_spec(m, torch, dev, stream, K=7, V=32768, n_sets=32, reps=8):
    """Acceptance of K = 7 drafts (a verify batch of 8 tokens) over a V = 32768 vocabulary (the hash-routed layers'
    vocabulary): n_sets seeded (p, q, drafts, u) sets, one call each, replayed reps times as a CUDA graph.
    The kernel reads one or two rows of V floats per call; its time is latency (one CTA, two block scans)."""
    from moe_inputs import spec_inputs
    sets = [spec_inputs(500 + i, K, V) for i in range(n_sets)]
    P = torch.from_numpy(np.stack([s[0] for s in sets])).to(dev)
    Q = torch.from_numpy(np.stack([s[1] for s in sets])).to(dev)
    D = torch.from_numpy(np.stack([s[2] for s in sets])).to(dev)
    U = torch.from_numpy(np.stack([s[3] for s in sets])).to(dev)
    R = torch.zeros((n_sets, 2), dtype=torch.int32, device=dev)

    def launch():
        for i in range(n_sets):
            m.moe_spec_accept(P[i], Q[i], K, V, D[i], U[i], R[i], stream=stream)
    with torch.cuda.stream(stream):
        launch()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        launch()
    with torch.cuda.stream(stream):
        g.replay()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    with torch.cuda.stream(stream):
        for _ in range(reps):
            g.replay()
    e1.record(stream)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1e3 / (reps * n_sets)
    kept = R[:, 0].float().mean().item()
    return {"workload": "acceptance of %d drafts, vocabulary %d, %d seeded sets" % (K, V, n_sets),
            "us_per_call": round(us, 3), "calls": reps * n_sets, "mean_kept": round(kept, 2),
            "gpu_launches_per_call": 1}


def bench_prefill(m, torch, args, dev, stream, layer_p, E):
    """Prefill grouped GEMM: args.prefill_tokens tokens, top-6 with Zipf(1.1) expert popularity, one call per step.
    Tensor roofline: useful FLOPs (pairs x 3 matrices x 2 H I) / call time against the fp8-rate tensor peak
    (measured bf16 dense peak x 2, the nominal fp8 / bf16 ratio; mxf8f6f4 MMAs run at the fp8 rate)."""
    from moe_inputs import x_bf16_bits, zipf_routing
    Tp = args.prefill_tokens
    xp = torch.from_numpy(x_bf16_bits(args.seed + 17, range(Tp), H).view(np.int16)).to(dev)
    ip, wp = zipf_routing(args.seed, Tp, E, K_TOP)
    idx_p = torch.from_numpy(ip).to(dev)
    w_p = torch.from_numpy(wp).to(dev)
    ws_p = layer_p.prefill_workspace(Tp, K_TOP, stream=stream)
    y_p = torch.empty((Tp, H), dtype=torch.float32, device=dev)
    yb_p = torch.empty((Tp, H), dtype=torch.int16, device=dev)

    def call():
        m.moe_expert_grouped_gemm_prefill(layer_p, xp, Tp, idx_p, w_p, K_TOP, y_p, yb_p, ws_p, stream=stream)

    for _ in range(max(3, args.warmup)):
        call()
    stream.synchronize()
    if m.moe_get_device_status(ws_p, stream) != 0:
        raise RuntimeError("device status after prefill warm-up")
    reps = max(3, args.steps)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(reps):
        call()
    e1.record(stream)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / reps
    if m.moe_get_device_status(ws_p, stream) != 0:
        raise RuntimeError("device status after prefill")
    counts = np.bincount(ip.reshape(-1), minlength=E)
    pairs = int(counts.sum())
    flops = pairs * 3 * 2.0 * H * I
    wbytes = int(np.count_nonzero(counts)) * (m.moe_packed_bytes(1, 1, 0, 1, H, I) + m.moe_packed_bytes(1, 1, 1, 1, H, I))
    peaks = measured_peaks()
    bf16 = peak_of(peaks, "bf16_tflops")
    peak = 2.0 * bf16 if bf16 else 3800.0
    hbm = peak_of(peaks, "hbm_gbs") or 6800.0
    tflops = flops / (ms * 1e-3) / 1e12
    return {"workload": "prefill of %d tokens, top-6, Zipf(1.1) expert popularity over %d experts (%d pairs, "
                        "%d tiles of 128)" % (Tp, E, pairs, int(np.sum((counts + 127) // 128))),
            "tok_s": round(Tp / (ms * 1e-3), 1), "ms_per_call": round(ms, 4), "calls": reps,
            "gpu_launches_per_call": 7,
            "roofline": {"bound": "tensor", "achieved": round(tflops, 1), "peak": round(peak, 1), "unit": "TFLOP/s",
                         "frac": round(tflops / peak, 4), "traffic": None,
                         "peak_source": ("MEASURED_PEAKS.json bf16_tflops x 2 (fp8 rate; of measured)" if bf16
                                         else "fallback 1900 bf16 x 2")},
            "weight_bytes": wbytes, "weight_gbs": round(wbytes / (ms * 1e-3) / 1e9, 1),
            "weight_frac_of_hbm": round(wbytes / (ms * 1e-3) / 1e9 / hbm, 4)}


# ------------------------------------------------------------------------------------------------ CPU oracle
class CpuOracle:
    """The oracle as it stands, on the host cores, for the first n tokens of the bench's workload (same seeds, same
    layer): its own routing of them, encoded experts per format (built once, before any timing), the timed sample
    of the CPU baseline and the parity check of the GPU's outputs."""

    def __init__(self, seed, n, n_experts=E):
        import oracle
        from moe_inputs import router_f16_bits, x_bf16_bits
        self.oracle = oracle
        self.seed = seed
        self.E = n_experts
        self.cores = os.cpu_count() or 1
        self.n = max(int(n), self.cores)
        wr = router_f16_bits(seed, 0, self.E, H)
        self.x = x_bf16_bits(seed, range(self.n), H)
        self.idx, self.w, self.logits, self.absl = oracle.route_topk(wr, self.x, K_TOP)
        self.enc = {}

    def _encode(self, fmt, experts):
        from moe_inputs import expert_matrix_f32
        todo = [(int(e), wh) for e in sorted(set(int(v) for v in np.ravel(experts))) for wh in range(3)
                if (fmt, int(e), wh) not in self.enc]

        def one(key):
            e, wh = key
            self.enc[(fmt, e, wh)] = self.oracle.encode(fmt, expert_matrix_f32(self.seed, 0, e, wh, H, I))
        with cf.ThreadPoolExecutor(self.cores) as ex:
            list(ex.map(one, todo))

    def _moe(self, fmt, idx, w, x):
        c = self.enc
        return self.oracle.moe_tokens(fmt, H, I, lambda e: c[(fmt, int(e), 0)], lambda e: c[(fmt, int(e), 1)],
                                      lambda e: c[(fmt, int(e), 2)], idx, w, x)

    def timed(self, fmt_name, seconds):
        """Tokens per second of the oracle, one token per thread, over the first `cores` tokens."""
        fmt = FMT_IDS[fmt_name]
        nt = self.cores
        self._encode(fmt, self.idx[:nt])
        done = 0
        t0 = time.time()
        with cf.ThreadPoolExecutor(self.cores) as ex:
            while time.time() - t0 < seconds or done == 0:
                list(ex.map(lambda t: self._moe(fmt, self.idx[t:t + 1], self.w[t:t + 1], self.x[t:t + 1]), range(nt)))
                done += nt
        el = time.time() - t0
        return {"value": round(done / el, 3), "unit": "tok/s", "cores": self.cores, "kind": "oracle",
                "sample": "%d tokens (%d per thread) of the same layer and routing rule in %.1f s wall; fp64 C oracle, "
                          "one token per thread" % (done, done // self.cores, el)}

    def _near_tie(self, t, got):
        """The GPU's top-k list of token t differs from the oracle's only by swaps of experts whose exact logits lie
        within the fp32 summation error bound of each other (H * 2^-24 * sum|terms| each)."""
        ref = self.idx[t]
        if np.array_equal(got, ref):
            return True
        lg, tol = self.logits[t], H * 2.0 ** -24 * self.absl[t]
        chosen = [int(e) for e in got]
        if len(set(chosen)) != K_TOP or min(chosen) < 0 or max(chosen) >= self.E:
            return False
        others = [e for e in range(self.E) if e not in chosen]
        for r in range(K_TOP):
            a = chosen[r]
            for b in chosen[r + 1:] + others:
                if lg[a] < lg[b] - (tol[a] + tol[b]):
                    return False
        return True

    def parity_shared(self, y_gpu, idx_gpu, w_gpu, sidx, yb_gpu):
        """Routed output (MXFP4, the GPU's routing) plus the Q8_0 shared expert sidx[t] (layer 1 of the same seed),
        against the GPU's combined y within 1e-3 * (sum|routed terms| + sum|shared terms|) + 1e-6; the bf16 copy
        equal to the round-to-nearest-even of y."""
        par = self.parity(1, y_gpu, idx_gpu, w_gpu, extra=lambda t: self._shared(int(sidx[t]), t))
        b = np.ascontiguousarray(y_gpu, np.float32).view(np.uint32).astype(np.uint64)
        rne = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
        par["bf16_copy_exact"] = bool(np.array_equal(rne, yb_gpu))
        par["ok"] = par["ok"] and par["bf16_copy_exact"]
        return par

    def _shared(self, e, t):
        from moe_inputs import expert_matrix_f32
        key = ("shared", e)
        if key not in self.enc:
            self.enc[key] = [self.oracle.encode(4, expert_matrix_f32(self.seed, 1, e, wh, H, I)) for wh in range(3)]
        gb, ub, db = self.enc[key]
        return self.oracle.moe_tokens(4, H, I, lambda _: gb, lambda _: ub, lambda _: db, np.zeros((1, 1), np.int32),
                                      np.ones((1, 1), np.float32), self.x[t:t + 1])

    def parity(self, fmt, y_gpu, idx_gpu, w_gpu, extra=None):
        """Compare the GPU's first tokens with the oracle: routing exactly (or up to proven near-ties), and y element
        by element within 1e-3 * sum|terms| + 1e-6 (the FFN of the GPU's own routing, so that a near-tie swap does
        not mask the FFN's check). NaN must match NaN."""
        n = len(y_gpu)
        exact = sum(int(np.array_equal(idx_gpu[t], self.idx[t])) for t in range(n))
        ties = sum(int(not np.array_equal(idx_gpu[t], self.idx[t]) and self._near_tie(t, idx_gpu[t])) for t in range(n))
        self._encode(fmt, idx_gpu)
        with cf.ThreadPoolExecutor(self.cores) as ex:
            res = list(ex.map(lambda t: self._moe(fmt, idx_gpu[t:t + 1], w_gpu[t:t + 1], self.x[t:t + 1]), range(n)))
        y_ref = np.concatenate([r[0] for r in res])
        ab = np.concatenate([r[1] for r in res])
        if extra is not None:   # a further term of every token's output (the shared expert), added in fp64
            for t in range(n):
                ye, abe = extra(t)
                y_ref[t] += ye[0]
                ab[t] += abe[0]
        y = np.asarray(y_gpu, dtype=np.float64)
        nan_ok = bool(np.array_equal(np.isnan(y), np.isnan(y_ref)))
        fin = ~np.isnan(y_ref)
        ratio = float(np.max(np.abs(y[fin] - y_ref[fin]) / (1e-3 * ab[fin] + 1e-6))) if fin.any() else 0.0
        ok = nan_ok and ratio <= 1.0 and exact + ties == n
        return {"tokens": n, "max_err_over_bound": round(ratio, 5), "routing_exact": exact, "routing_near_ties": ties,
                "tolerance": "|y - y_oracle| <= 1e-3 * sum|terms| + 1e-6 per element", "ok": ok}


def main():
    args = parse()
    if args.impl == "reference":
        rank = int(os.environ.get("RANK", "0"))
        if rank != 0:
            return
        t0 = time.time()
        per_step = max(2.0, 60.0 / max(1, args.steps + args.warmup))
        co = CpuOracle(args.seed, 0, args.experts)
        for _ in range(args.warmup):
            co.timed(args.fmt, per_step / 4)
        vals = [co.timed(args.fmt, per_step) for _ in range(args.steps)]
        v = float(np.median([r["value"] for r in vals]))
        cb = dict(vals[0])
        cb["value"] = v
        out = {"impl": "reference", "metric": "routed-MoE decode tok/s and HBM GB/s (% of 8 TB/s), MXFP4/Q2_K/INT4 experts",
               "value": v, "unit": "tok/s", "n_gpus": 0, "steps": args.steps, "warmup": args.warmup,
               "ms_per_step": None, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
               "dtype": "f64", "data": "synthetic",
               "config": {"workload": "DS4-Flash routed-MoE layer decode, batch 1, sampled tokens", "H": H, "I": I,
                          "experts": E, "top_k": K_TOP, "format": args.fmt},
               "cpu_baseline": cb, "e2e": {"value": v, "unit": "tok/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
               "wall_s": round(time.time() - t0, 1)}
        print(json.dumps(out))
        return
    out, checks = run_ours(args)
    if out is None:
        return
    single = int(os.environ.get("WORLD_SIZE", "1")) == 1
    breach = False
    if single and (checks or not args.no_cpu_baseline):
        co = CpuOracle(args.seed, max([len(c[2]) for c in checks] + [0]), args.experts)
        for key, fmt, y_rows, idx_rows, w_rows, *more in checks:
            if key == "shared_expert":
                par = co.parity_shared(y_rows, idx_rows, w_rows, *more)
                out["shared_expert"]["parity"] = par
            else:
                par = co.parity(fmt, y_rows, idx_rows, w_rows)
                if key is None:
                    out["parity"] = par
                else:
                    out["formats"][key]["parity"] = par
            breach |= not par["ok"]
        if not args.no_cpu_baseline:
            out["cpu_baseline"] = co.timed(args.fmt, args.cpu_seconds)
    print(json.dumps(out))
    if breach:
        sys.exit(1)


if __name__ == "__main__":
    main()
