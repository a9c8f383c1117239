#!/usr/bin/env python
"""Throughput of the fused 4-bit block-scaled MoE layer on GB300.

One step = one moe_forward pass (routing, align/permute, grouped GEMM1 +
activation, grouped GEMM2 + routing weight, unpermute) over one batch of
synthetic input of the chosen workload (default: the gpt-oss-20b-shaped
decode layer, T=64 E=32 top-4 H=I=2880 NVFP4). Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config c1]
  python bench.py --impl reference ...   # the CPU oracle on the host cores

With N > 1 (torchrun) every rank runs an independent replica of the layer on
its own GPU (the path has no exchange step) and rank 0 reports the aggregate.
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

L2_FLUSH_BYTES = 256 << 20  # larger than the 129 MB L2


def algorithmic_bytes(cfg, ids=None):
    """Bytes the layer must move at minimum: active experts' packed weights,
    block scales, global scales and biases, plus x, out, logits, ids/weights."""
    per_w = {"nvfp4": 0.5 + 1 / 16, "mxfp4": 0.5 + 1 / 32, "int4": 0.5 + 2 / 64 + 0.5 / 64}[cfg.fmt]

    def proj(N, K):
        b = N * K * per_w + (4 if cfg.fmt == "nvfp4" else 0)
        if cfg.bias:
            b += N * 2
        return b

    if ids is None:
        active = min(cfg.E, cfg.T * cfg.k)
    else:
        active = len(set(int(i) for i in ids.reshape(-1)))
    w13 = proj(cfg.N1, cfg.H)
    w2 = proj(cfg.H, cfg.I)
    act = 2 * cfg.T * cfg.H * 2 + cfg.T * cfg.E * 4 + cfg.T * cfg.k * 8
    return dict(total=active * (w13 + w2) + act, w13=active * w13, w2=active * w2, active=active)


def algorithmic_flops(cfg):
    return 2 * cfg.T * cfg.k * (cfg.N1 * cfg.H + cfg.H * cfg.I)


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except Exception:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def gemm_source_hash():
    """Hash of what defines the grouped GEMM kernel (its source, the device
    helpers it includes and its argument struct), recorded beside each ncu
    summary: a summary whose hash differs was taken on other GEMM code."""
    import hashlib
    import re
    csrc = os.path.join(ROOT, "bit_block_scaled_gb300", "csrc")
    h = hashlib.sha256()
    for f in ("gemm.cu", "common.cuh", "dequant.cuh"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(fh.read())
    with open(os.path.join(csrc, "kernels.h")) as fh:
        args = re.search(r"struct GemmArgs \{.*?\};", fh.read(), flags=re.S)
    h.update(args.group(0).encode())
    return h.hexdigest()[:16]


def operand_dtype(cfg):
    """The tensor-core operand type each GEMM of the fused forward uses.
    NVFP4 expands exactly to f16 (E2M1 value times E4M3 scale); its GEMM1 runs
    on f16 operands, and GEMM2 too when the activation is swigluoai. The other
    formats dequantise to bf16. Accumulation is fp32 throughout."""
    if cfg.fmt == "nvfp4":
        g2 = "f16" if cfg.act == "swigluoai" else "bf16"
        return f"GEMM1 f16 / GEMM2 {g2} operands (4-bit weights dequantised), fp32 accumulate"
    return "bf16 operands (4-bit weights dequantised), fp32 accumulate"


def read_traffic(kernel_tag):
    """DRAM bytes per launch of the kernel from the committed ncu summary, if
    it was captured for the current kernel source (else None)."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.txt")
    try:
        vals = {}
        with open(path) as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    vals[k.strip()] = v.strip()
        if vals.get("source_hash") != gemm_source_hash():
            return None, vals.get("source_hash")
        return float(vals["traffic_bytes_per_launch"]), vals.get("source_hash")
    except Exception:
        return None, None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.samples = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.idx}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 8:
                self.samples.append((time.time(), parts))

    def stop(self):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self, t0, t1):
        sel = [p for (t, p) in self.samples if t0 - 0.25 <= t <= t1 + 0.25]
        if not sel:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        sm = [float(p[0]) for p in sel if p[0].replace(".", "").isdigit()]
        mx = [float(p[1]) for p in sel if p[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for p in sel:
            for name, v in zip(names, p[4:8]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sel)}


def rejected(clocks):
    bad = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}
    if bad & set(clocks.get("reasons", [])):
        return True
    sm, mx = clocks.get("sm_mhz"), clocks.get("sm_max_mhz")
    return bool(sm and mx and sm < 0.5 * mx and not clocks.get("reasons"))


def reduce_max_over_ranks(pg, values, device):
    """Max over ranks of each per-rank duration: the slowest replica sets the
    job's time. pg is torch.distributed (initialised) or None for one rank."""
    import torch
    if pg is None:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], device=device, dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t]


def job_tokens_per_s(world, tokens_per_step, steps, total_ms):
    """Whole-job throughput: every replica processes tokens_per_step per step."""
    return world * tokens_per_step * steps / (total_ms / 1e3)


def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


# --------------------------------------------------------------- our arm (GPU)
def run_ours(args):
    import torch
    import bit_block_scaled_gb300 as moe
    from bit_block_scaled_gb300 import build as _build
    from synth import get_config, make_layer

    rank, world, local = dist_env()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist
    if rank == 0 or not os.path.exists(moe._lib.LIB_PATH):
        _build.build()
    if pg:
        pg.barrier()
    moe.load()
    cfg = get_config(args.config)
    L = make_layer(cfg, seed=args.seed, device="cuda")
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    bm = args.block_m
    nbytes = moe.moe_workspace_size(T, E, k, H, I, bm)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device="cuda")
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    q13, q2 = moe.qweight(L["w13"]), moe.qweight(L["w2"])
    act = moe.act(cfg.act, cfg.alpha, cfg.limit)
    route = moe.ROUTE[cfg.route]
    stream = torch.cuda.Stream()

    def fwd():
        moe.moe_forward(L["x"], L["logits"], L["sel_bias"], k, route, q13, q2, 0, act, 1, bm, out, ws,
                        stream)

    with torch.cuda.stream(stream):
        for _ in range(3):
            fwd()
    torch.cuda.synchronize()
    launches_per_step = moe.moe_last_launch_count()
    # capture one forward in a CUDA graph (the layer as a serving loop runs it)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        with torch.cuda.graph(graph, stream=stream):
            fwd()
    torch.cuda.synchronize()
    moe.moe_clear_status(ws, stream)

    def timed_loop(n, run):
        starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
        with torch.cuda.stream(stream):
            for i in range(n):
                flush.zero_()               # evict L2 (untimed)
                starts[i].record(stream)
                run()
                ends[i].record(stream)
        torch.cuda.synchronize()
        return [s.elapsed_time(e) for s, e in zip(starts, ends)]

    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    bus = getattr(props, "pci_bus_id", None)
    sampler = ClockSampler(f"{getattr(props, 'pci_domain_id', 0):08x}:{bus:02x}:"
                           f"{getattr(props, 'pci_device_id', 0):02x}.0" if bus is not None else local)
    sampler.start()
    time.sleep(0.3)
    timed_loop(args.warmup, graph.replay)
    for attempt in range(2):
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        times = timed_loop(args.steps, graph.replay)
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        t1 = time.time()
        time.sleep(0.2)
        clocks = sampler.summary(t0, t1)
        if not rejected(clocks):
            break
    sampler.stop()
    total_ms = sum(times)
    st = moe.moe_read_status(ws, stream)
    if st != 0:
        raise SystemExit(f"device status {moe.moe_status_string(st)}")

    # per-kernel breakdown: each step entry point timed with events on the stream
    bd = breakdown(moe, L, cfg, bm, stream, flush, args.breakdown_iters)

    # end to end through the C ABI with host buffers (pinned), copies inside
    xh = L["x"].cpu().pin_memory()
    lh = L["logits"].cpu().pin_memory()
    oh = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()

    def e2e():
        moe.moe_forward_host(xh, lh, L["sel_bias"], k, route, q13, q2, 0, act, 1, bm, oh, ws, stream)

    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            e2e()
    torch.cuda.synchronize()
    e2e_times = []
    for _ in range(args.e2e_steps):
        flush.zero_()
        torch.cuda.synchronize()
        s_ev, e_ev = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s_ev.record(stream)
        e2e()
        e_ev.record(stream)
        e_ev.synchronize()
        e2e_times.append(s_ev.elapsed_time(e_ev))

    total_ms, e2e_total = reduce_max_over_ranks(pg, [total_ms, sum(e2e_times)], "cuda")
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return
    ms = total_ms / args.steps
    value = job_tokens_per_s(world, T, args.steps, total_ms)
    e2e_ms = e2e_total / len(e2e_times)
    ids = None
    try:
        ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
        tw = torch.empty(T, k, dtype=torch.float32, device="cuda")
        moe.moe_route_topk(L["logits"], L["sel_bias"], k, route, ids, tw, ws, stream)
        torch.cuda.synchronize()
        ids = ids.cpu().numpy()
    except Exception:
        ids = None
    ab = algorithmic_bytes(cfg, ids)
    flops = algorithmic_flops(cfg)
    peaks, peak_src = read_peaks()
    hbm = peaks["hbm_gbs"]
    tc = peaks["bf16_tflops"]
    gemm1_ms = bd["gemm1_ms"]
    decode = flops / (tc * 1e12) < ab["total"] / (hbm * 1e9)
    if decode:
        g1_bytes = ab["w13"] + cfg.T * cfg.k * (cfg.H + cfg.I) * 2
        achieved = g1_bytes / (gemm1_ms / 1e3) / 1e9
        traffic, _ = read_traffic(f"gemm1_{args.config}")
        roofline = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                    "frac": round(achieved / hbm, 4), "traffic": traffic,
                    "kernel": "grouped_gemm_kernel (GEMM1 + act)", "peak_source": peak_src,
                    "algorithmic_bytes_per_launch": int(g1_bytes)}
    else:
        g1_flops = 2 * cfg.T * cfg.k * cfg.N1 * cfg.H
        achieved = g1_flops / (gemm1_ms / 1e3) / 1e12
        traffic, _ = read_traffic(f"gemm1_{args.config}")
        roofline = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tc, "unit": "TFLOP/s",
                    "frac": round(achieved / tc, 4), "traffic": traffic,
                    "kernel": "grouped_gemm_kernel (GEMM1 + act)", "peak_source": peak_src,
                    "algorithmic_flops_per_launch": int(g1_flops)}
    layer_frac = max(ab["total"] / (hbm * 1e9), flops / (tc * 1e12)) / (ms / 1e3)
    rec = {
        "metric": "MoE-layer tokens/s on 1 GB300; % of HBM BW (decode) / bf16 TC peak (prefill)",
        "value": round(value, 1),
        "unit": "tokens/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": operand_dtype(cfg),
        "data": "synthetic (seeded; weights N(0,0.02) quantised per the workload recipe)",
        "config": {"workload": cfg.workload, "name": args.config, "T": T, "E": E, "top_k": k, "H": H,
                   "I": I, "format": cfg.fmt, "activation": cfg.act, "block_m": bm,
                   "parallelism": f"replicas x{world}", "l2": "flushed (256 MiB write) before every step",
                   "launch": "CUDA graph of one moe_forward"},
        "layer_roofline_frac": round(layer_frac, 4),
        "algorithmic_bytes": int(ab["total"]),
        "algorithmic_flops": int(flops),
        "breakdown_ms": {k2: round(v, 5) for k2, v in bd.items()},
        "roofline": roofline,
        "e2e": {"value": round(job_tokens_per_s(world, T, 1, e2e_ms), 1), "unit": "tokens/s",
                "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": int(T * H * 2 + T * E * 4), "d2h_bytes_per_step": int(T * H * 2)},
        "gpu_launches": int(launches_per_step * args.steps),
        "clocks": clocks,
    }
    if not args.no_cpu_baseline and world == 1:
        rec["cpu_baseline"] = cpu_baseline(cfg, L, args)
    print(json.dumps(rec), flush=True)
    if pg:
        pg.destroy_process_group()


def breakdown(moe, L, cfg, bm, stream, flush, iters):
    """Median device time of each of moe_forward's six kernels, as the forward
    runs them (moe_forward_profile: CUDA events around each launch on the
    stream; L2 flushed before each pass)."""
    import torch
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    ws = torch.zeros(moe.moe_workspace_size(T, E, k, H, I, bm), dtype=torch.uint8, device="cuda")
    out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
    act = moe.act(cfg.act, cfg.alpha, cfg.limit)
    q13, q2 = moe.qweight(L["w13"]), moe.qweight(L["w2"])
    route = moe.ROUTE[cfg.route]
    res = {}
    with torch.cuda.stream(stream):
        for it in range(iters + 3):
            flush.zero_()
            ms = moe.moe_forward_profile(L["x"], L["logits"], L["sel_bias"], k, route, q13, q2, 0, act, 1, bm,
                                         out, ws, stream)
            if it >= 3:
                for name, v in ms.items():
                    res.setdefault(name, []).append(v)
    med = {name: statistics.median(v) for name, v in res.items()}
    return {"route_ms": med["route"], "align_gather_ms": med["align"] + med["gather"],
            "gemm1_ms": med["gemm1"], "gemm2_ms": med["gemm2"], "unpermute_ms": med["unpermute"]}


# ---------------------------------------------------------- the CPU oracle
def oracle_step_sample(cfg, N, tokens):
    """One oracle pass (routing, align, GEMMs, unpermute) over a token sample."""
    from oracle import layer as OL
    from oracle import routing as OR
    sl = list(tokens)
    return OL.moe_forward(N["x"][sl], N["logits"][sl], N["w13"], N["w2"], cfg.k,
                          route_mode=OR.ROUTE_TOPK_SOFTMAX if cfg.route == "topk_softmax"
                          else OR.ROUTE_SIGMOID_BIAS, sel_bias=N.get("sel_bias"),
                          act=OL.ACT_SWIGLUOAI if cfg.act == "swigluoai" else OL.ACT_RELU2,
                          alpha=cfg.alpha, limit=cfg.limit)


def cpu_baseline(cfg, L, args, budget_s=20.0):
    from synth import to_numpy
    N = to_numpy(L)
    cores = len(os.sched_getaffinity(0))
    t0 = time.time()
    done = 0
    t = 0
    while time.time() - t0 < budget_s and done < cfg.T:
        oracle_step_sample(cfg, N, [t % cfg.T])
        done += 1
        t += 1
    el = time.time() - t0
    return {"value": round(done / el, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{done} token(s) of {args.config}, one oracle moe_forward per token "
                      f"(float64 NumPy, full dequantisation of the routed experts each call)"}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    from synth import get_config, make_layer, to_numpy
    cfg = get_config(args.config)
    N = to_numpy(make_layer(cfg, seed=args.seed, device="cpu"))
    cores = len(os.sched_getaffinity(0))
    budget = args.ref_budget_s
    t_start = time.time()
    for i in range(args.warmup):
        oracle_step_sample(cfg, N, [i % cfg.T])
        if time.time() - t_start > budget * 0.25:
            break
    times = []
    t0 = time.time()
    for i in range(args.steps):
        s = time.time()
        oracle_step_sample(cfg, N, [i % cfg.T])
        times.append(time.time() - s)
        if time.time() - t0 > budget:
            break
    total = sum(times)
    value = len(times) / total
    rec = {
        "metric": "MoE-layer tokens/s on 1 GB300; % of HBM BW (decode) / bf16 TC peak (prefill)",
        "impl": "reference",
        "value": round(value, 4), "unit": "tokens/s", "n_gpus": world, "steps": len(times),
        "steps_requested": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 accumulate (NumPy oracle)",
        "data": "synthetic (seeded)",
        "config": {"workload": cfg.workload, "name": args.config, "T": cfg.T, "E": cfg.E,
                   "top_k": cfg.k, "H": cfg.H, "I": cfg.I, "format": cfg.fmt,
                   "parallelism": "host cores, rank 0 only"},
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "sample": "one token of the workload per step through the oracle's moe_forward; "
                                   f"run capped at {budget:.0f} s"},
        "e2e": {"value": round(value, 4), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(rec), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--config", default="c1")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--block-m", type=int, default=16)
    ap.add_argument("--breakdown-iters", type=int, default=20)
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ref-budget-s", type=float, default=150.0)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
