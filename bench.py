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


def workload_config(cfg, args, world):
    """The `config` object of the JSON line; both arms print the same one."""
    return {"workload": cfg.workload, "name": args.config, "T": cfg.T, "E": cfg.E, "top_k": cfg.k,
            "H": cfg.H, "I": cfg.I, "format": cfg.fmt, "activation": cfg.act, "route": cfg.route,
            "block_m": args.block_m, "parallelism": f"replicas x{world}",
            "l2": "flushed (256 MiB write) before every GPU step"}


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
_PROJ_CACHE = {}


def layer_for(cfg, seed, device):
    """make_layer, with each projection made once per base workload and seed
    (the c3 sweep's three token counts share one set of weights)."""
    from synth.gen import make_activations, make_projection
    d = make_activations(cfg, seed, device)
    base = cfg.name.split("_t")[0]
    for which, N, K in (("w13", cfg.N1, cfg.H), ("w2", cfg.H, cfg.I)):
        key = (base, which, seed, device)
        if key not in _PROJ_CACHE:
            _PROJ_CACHE[key] = make_projection(cfg, which, N, K, seed, device, cfg.bias)
        d[which] = _PROJ_CACHE[key]
    d["cfg"] = cfg
    return d


class Layer:
    """One workload's inputs, workspace and output on the device, plus a CUDA
    graph of one moe_forward over them."""

    def __init__(self, moe, cfg, seed, block_m, stream):
        import torch
        self.moe, self.cfg, self.bm, self.stream = moe, cfg, block_m, stream
        self.L = layer_for(cfg, seed, "cuda")
        T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
        self.ws = torch.zeros(moe.moe_workspace_size(T, E, k, H, I, block_m), dtype=torch.uint8, device="cuda")
        self.out = torch.empty(T, H, dtype=torch.bfloat16, device="cuda")
        self.q13, self.q2 = moe.qweight(self.L["w13"]), moe.qweight(self.L["w2"])
        self.act = moe.act(cfg.act, cfg.alpha, cfg.limit)
        self.route = moe.ROUTE[cfg.route]
        with torch.cuda.stream(stream):
            for _ in range(3):
                self.fwd()
        torch.cuda.synchronize()
        self.launches = moe.moe_last_launch_count()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(stream):
            with torch.cuda.graph(self.graph, stream=stream):
                self.fwd()
        torch.cuda.synchronize()
        moe.moe_clear_status(self.ws, stream)

    def fwd(self):
        L = self.L
        self.moe.moe_forward(L["x"], L["logits"], L["sel_bias"], self.cfg.k, self.route, self.q13, self.q2, 0,
                             self.act, 1, self.bm, self.out, self.ws, self.stream)

    def status(self):
        return self.moe.moe_read_status(self.ws, self.stream)

    def routing_ids(self):
        import torch
        cfg = self.cfg
        ids = torch.empty(cfg.T, cfg.k, dtype=torch.int32, device="cuda")
        tw = torch.empty(cfg.T, cfg.k, dtype=torch.float32, device="cuda")
        ws = torch.zeros(self.moe._lib.STATUS_BYTES, dtype=torch.uint8, device="cuda")
        self.moe.moe_route_topk(self.L["logits"], self.L["sel_bias"], cfg.k, self.route, ids, tw, ws, self.stream)
        torch.cuda.synchronize()
        return ids.cpu().numpy()


def timed_loop(stream, flush, n, run):
    """n steps, each timed with CUDA events on `stream`; L2 flushed (untimed)
    before every step. Returns the per-step device times in ms."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    with torch.cuda.stream(stream):
        for i in range(n):
            flush.zero_()
            starts[i].record(stream)
            run()
            ends[i].record(stream)
    torch.cuda.synchronize()
    return [s_.elapsed_time(e) for s_, e in zip(starts, ends)]


def breakdown(layer, flush, iters):
    """Median device time of each of moe_forward's six kernels, as the forward
    runs them (moe_forward_profile: CUDA events around each launch on the
    stream; L2 flushed before each pass)."""
    import torch
    moe, cfg, L = layer.moe, layer.cfg, layer.L
    res = {}
    with torch.cuda.stream(layer.stream):
        for it in range(iters + 3):
            flush.zero_()
            ms = moe.moe_forward_profile(L["x"], L["logits"], L["sel_bias"], cfg.k, layer.route, layer.q13,
                                         layer.q2, 0, layer.act, 1, layer.bm, layer.out, layer.ws, layer.stream)
            if it >= 3:
                for name, v in ms.items():
                    res.setdefault(name, []).append(v)
    med = {name: statistics.median(v) for name, v in res.items()}
    return {"route_ms": med["route"], "align_gather_ms": med["align"] + med["gather"],
            "gemm1_ms": med["gemm1"], "gemm2_ms": med["gemm2"], "unpermute_ms": med["unpermute"]}


def roofline_of(cfg, ids, ms_layer, bd, peaks, peak_src, args_config):
    """Roofline of the dominant kernel (GEMM1) and of the whole layer: HBM for
    decode shapes (bytes bound), bf16 tensor peak for prefill shapes."""
    ab = algorithmic_bytes(cfg, ids)
    flops = algorithmic_flops(cfg)
    hbm, tc = peaks["hbm_gbs"], peaks["bf16_tflops"]
    decode = flops / (tc * 1e12) < ab["total"] / (hbm * 1e9)
    g1 = bd["gemm1_ms"] / 1e3
    traffic, _ = read_traffic(f"gemm1_{args_config}")
    if decode:
        g1_bytes = ab["w13"] + cfg.T * cfg.k * (cfg.H + cfg.I) * 2
        achieved = g1_bytes / g1 / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                "frac": round(achieved / hbm, 4), "traffic": traffic,
                "kernel": "grouped_gemm_kernel (GEMM1 + act)", "peak_source": peak_src,
                "algorithmic_bytes_per_launch": int(g1_bytes)}
        layer_frac = ab["total"] / (hbm * 1e9) / (ms_layer / 1e3)
    else:
        g1_flops = 2 * cfg.T * cfg.k * cfg.N1 * cfg.H
        achieved = g1_flops / g1 / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": tc, "unit": "TFLOP/s",
                "frac": round(achieved / tc, 4), "traffic": traffic,
                "kernel": "grouped_gemm_kernel (GEMM1 + act)", "peak_source": peak_src,
                "algorithmic_flops_per_launch": int(g1_flops)}
        layer_frac = flops / (tc * 1e12) / (ms_layer / 1e3)
    return roof, layer_frac, ab, flops, decode


# the other workloads, each timed in the same run (the default workload is the
# headline line); they are parity cases too
OTHER_WORKLOADS = ("c2", "c3_t1", "c3_t32", "c3_t8192", "c4")


def measure_other(moe, key, args, stream, flush, peaks, peak_src):
    import torch
    from synth import get_config
    cfg = get_config(key)
    layer = Layer(moe, cfg, args.seed, args.block_m, stream)
    timed_loop(stream, flush, max(args.warmup, 3), layer.graph.replay)
    times = timed_loop(stream, flush, args.workload_steps, layer.graph.replay)
    st = layer.status()
    if st != 0:
        raise SystemExit(f"{key}: device status {moe.moe_status_string(st)}")
    ms = statistics.median(times)
    bd = breakdown(layer, flush, max(5, args.breakdown_iters // 2))
    roof, layer_frac, ab, flops, decode = roofline_of(cfg, layer.routing_ids(), ms, bd, peaks, peak_src, key)
    rec = {"workload": cfg.workload, "tokens_per_s": round(cfg.T / (ms / 1e3), 1), "ms_per_step": round(ms, 5),
           "steps": len(times), "bound": roof["bound"], "layer_roofline_frac": round(layer_frac, 4),
           "gemm1_frac": roof["frac"], "gemm1_ms": round(bd["gemm1_ms"], 5), "gemm2_ms": round(bd["gemm2_ms"], 5),
           "breakdown_ms": {k2: round(v, 5) for k2, v in bd.items()},
           "peak": roof["peak"], "peak_unit": roof["unit"], "active_experts": ab["active"],
           "algorithmic_bytes": int(ab["total"]), "algorithmic_flops": int(flops),
           "gpu_launches_per_step": layer.launches, "dtype": operand_dtype(cfg)}
    del layer
    torch.cuda.empty_cache()
    return rec


def run_ours(args):
    import torch
    import bit_block_scaled_gb300 as moe
    from bit_block_scaled_gb300 import build as _build
    from synth import get_config

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
    T, E, k, H, I = cfg.T, cfg.E, cfg.k, cfg.H, cfg.I
    bm = args.block_m
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.Stream()
    layer = Layer(moe, cfg, args.seed, bm, stream)
    L = layer.L

    props = torch.cuda.get_device_properties(torch.cuda.current_device())
    bus = getattr(props, "pci_bus_id", None)
    sampler = ClockSampler(f"{getattr(props, 'pci_domain_id', 0):08x}:{bus:02x}:"
                           f"{getattr(props, 'pci_device_id', 0):02x}.0" if bus is not None else local)
    sampler.start()
    time.sleep(0.3)
    timed_loop(stream, flush, args.warmup, layer.graph.replay)
    for attempt in range(2):
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        t0 = time.time()
        times = timed_loop(stream, flush, args.steps, layer.graph.replay)
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
    st = layer.status()
    if st != 0:
        raise SystemExit(f"device status {moe.moe_status_string(st)}")

    # per-kernel breakdown: moe_forward_profile's events around each launch
    bd = breakdown(layer, flush, args.breakdown_iters)

    # end to end through the C ABI with host buffers (pinned: the kernels read
    # x and logits and write out over the host link inside the timed region)
    xh = L["x"].cpu().pin_memory()
    lh = L["logits"].cpu().pin_memory()
    oh = torch.empty(T, H, dtype=torch.bfloat16).pin_memory()

    def e2e():
        moe.moe_forward_host(xh, lh, L["sel_bias"], k, layer.route, layer.q13, layer.q2, 0, layer.act, 1, bm, oh,
                             layer.ws, stream)

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
    peaks, peak_src = read_peaks()
    roofline, layer_frac, ab, flops, _ = roofline_of(cfg, layer.routing_ids(), ms, bd, peaks, peak_src,
                                                     args.config)
    launches = layer.launches
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
        "data": "synthetic (seeded CPU generators; weights N(0,0.02) quantised per the workload recipe)",
        "config": workload_config(cfg, args, world),
        "launch": "CUDA graph of one moe_forward per step",
        "layer_roofline_frac": round(layer_frac, 4),
        "algorithmic_bytes": int(ab["total"]),
        "algorithmic_flops": int(flops),
        "breakdown_ms": {k2: round(v, 5) for k2, v in bd.items()},
        "roofline": roofline,
        "e2e": {"value": round(job_tokens_per_s(world, T, 1, e2e_ms), 1), "unit": "tokens/s",
                "ms_per_step": round(e2e_ms, 5),
                "h2d_bytes_per_step": int(T * H * 2 + T * E * 4), "d2h_bytes_per_step": int(T * H * 2)},
        "gpu_launches": int(launches * args.steps),
        "clocks": clocks,
    }
    del layer
    torch.cuda.empty_cache()
    if not args.no_workloads and world == 1:
        rec["workloads"] = {key: measure_other(moe, key, args, stream, flush, peaks, peak_src)
                            for key in OTHER_WORKLOADS if key != args.config}
    if not args.no_cpu_baseline and world == 1:
        rec["cpu_baseline"] = cpu_baseline(cfg, args)
    print(json.dumps(rec), flush=True)
    if pg:
        pg.destroy_process_group()


# ---------------------------------------------------------- the CPU oracle
def oracle_batch(cfg, N, acc_dtype):
    """One oracle pass (routing, align, GEMMs streamed per expert, unpermute)
    over the whole batch of the workload."""
    import numpy as np
    from oracle import layer as OL
    from oracle import routing as OR
    return OL.moe_forward(N["x"], N["logits"], N["w13"], N["w2"], cfg.k,
                          route_mode=OR.ROUTE_TOPK_SOFTMAX if cfg.route == "topk_softmax"
                          else OR.ROUTE_SIGMOID_BIAS, sel_bias=N.get("sel_bias"),
                          act=OL.ACT_SWIGLUOAI if cfg.act == "swigluoai" else OL.ACT_RELU2,
                          alpha=cfg.alpha, limit=cfg.limit, acc_dtype=np.dtype(acc_dtype))


def oracle_layer_numpy(cfg, seed):
    """Host NumPy copy of the workload, with only the routed experts' weights
    drawn (the oracle never reads the others)."""
    import numpy as np
    from oracle import routing as OR
    from synth import to_numpy
    from synth.gen import make_activations, make_projection
    d = make_activations(cfg, seed, "cpu")
    logits = d["logits"].numpy()
    if cfg.route == "topk_softmax":
        ids, _ = OR.topk_softmax(logits, cfg.k)
    else:
        ids, _ = OR.sigmoid_bias_topk(logits, d["sel_bias"].numpy(), cfg.k)
    experts = sorted(set(int(e) for e in np.unique(ids)))
    d["w13"] = make_projection(cfg, "w13", cfg.N1, cfg.H, seed, "cpu", cfg.bias, experts=experts)
    d["w2"] = make_projection(cfg, "w2", cfg.H, cfg.I, seed, "cpu", cfg.bias, experts=experts)
    d["cfg"] = cfg
    return to_numpy(d), len(experts)


def oracle_child(args):
    """Child process of the CPU baseline (BLAS threads fixed by its
    environment): times one float32-accumulate oracle pass over the whole
    batch of each named workload and prints one JSON object."""
    from synth import get_config
    res = {}
    for key in args.oracle_child.split(","):
        cfg = get_config(key)
        N, active = oracle_layer_numpy(cfg, args.seed)
        t0 = time.perf_counter()
        oracle_batch(cfg, N, "float32")
        el = time.perf_counter() - t0
        res[key] = {"tokens_per_s": round(cfg.T / el, 4), "seconds": round(el, 3), "tokens": cfg.T,
                    "active_experts": active}
    print(json.dumps(res), flush=True)


def _run_oracle_child(keys, threads, seed):
    env = dict(os.environ)
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        env[var] = str(threads)
    env["CUDA_VISIBLE_DEVICES"] = ""
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", ",".join(keys),
                        "--seed", str(seed)], env=env, capture_output=True, text=True, timeout=900)
    if r.returncode != 0:
        raise SystemExit("oracle child failed: " + r.stderr[-2000:])
    return json.loads([l for l in r.stdout.splitlines() if l.startswith("{")][-1])


def cpu_baseline(cfg, args):
    """The oracle in float32-accumulate mode over the whole batch of the
    workload (experts streamed one at a time), on all the host cores; plus
    one-thread figures for the tiny layer, the decode layer and the
    one-token MXFP4 layer."""
    cores = len(os.sched_getaffinity(0))
    main = _run_oracle_child([args.config], cores, args.seed)[args.config]
    one = _run_oracle_child(["c0", "c1", "c3_t1"], 1, args.seed)
    return {"value": main["tokens_per_s"], "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "mode": "float32 accumulate, whole batch, experts streamed one at a time",
            "sample": f"one oracle pass over all {main['tokens']} tokens of {args.config} "
                      f"({main['active_experts']} routed experts dequantised once each), "
                      f"{main['seconds']} s, BLAS threads = {cores}",
            "one_thread": {k2: v["tokens_per_s"] for k2, v in one.items()}}


def run_reference(args):
    rank, world, local = dist_env()
    if rank != 0:
        return
    import numpy as np
    from synth import get_config
    cfg = get_config(args.config)
    N, active = oracle_layer_numpy(cfg, args.seed)
    cores = len(os.sched_getaffinity(0))
    budget = args.ref_budget_s
    t_start = time.time()
    for i in range(args.warmup):
        oracle_batch(cfg, N, np.float32)
        if time.time() - t_start > budget * 0.25:
            break
    times = []
    t0 = time.time()
    for i in range(args.steps):
        s_ = time.perf_counter()
        oracle_batch(cfg, N, np.float32)
        times.append(time.perf_counter() - s_)
        if time.time() - t0 > budget:
            break
    total = sum(times)
    value = cfg.T * len(times) / total
    rec = {
        "metric": "MoE-layer tokens/s on 1 GB300; % of HBM BW (decode) / bf16 TC peak (prefill)",
        "impl": "reference",
        "value": round(value, 4), "unit": "tokens/s", "n_gpus": world, "steps": len(times),
        "steps_requested": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * total / len(times), 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32 accumulate (NumPy oracle)",
        "data": "synthetic (seeded CPU generators)",
        "config": workload_config(cfg, args, world),
        "cpu_baseline": {"value": round(value, 4), "unit": "tokens/s", "cores": cores, "kind": "oracle",
                         "mode": "float32 accumulate, whole batch, experts streamed one at a time",
                         "sample": f"each step one oracle pass over all {cfg.T} tokens of {args.config} "
                                   f"({active} routed experts); run capped at {budget:.0f} s"},
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
    ap.add_argument("--workload-steps", type=int, default=100)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true")
    ap.add_argument("--ref-budget-s", type=float, default=150.0)
    ap.add_argument("--oracle-child", default=None, help=argparse.SUPPRESS)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    if args.oracle_child:
        oracle_child(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
