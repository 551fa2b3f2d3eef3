"""Benchmark of the NVFP4 MoE layer (decode) on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload decode_c16|decode_b512|wide|tiny|gemm_sweep]
                    [--mode w4a4|w4a16|mxw4a4|w4a8] [--router] [--sweep-ms M,...]

Prints ONE JSON line (rank 0).  A step is one full MoE layer forward over the
workload's batch -- route/permute + activation quantisation -> gate_up
grouped GEMM -> SwiGLU+requant -> down grouped GEMM -> combine -- as one
moe_layer_forward call through the C ABI.  The timed region is one replay of
a CUDA graph holding K such calls.  The dominant kernel's duration (the
gate_up grouped GEMM, for the roofline figure) comes from a second graph of
the same K steps through the staged entry points with CUDA events around
every gate_up launch.  `e2e` replays moe_layer_forward_host (inputs read from
and output written to pinned host memory) once per step with a host
synchronisation.  Weights are random N(0, 0.02) quantised on the GPU;
activations N(0, 1) bf16; routing logits per the workload recipe.  Touched
weights per step exceed the 129 MB L2 by an order of magnitude, so no L2
flush is needed between steps.  --router times the router-logits GEMM and
--workload gemm_sweep the single-expert GEMM sweep instead.

At N=1 the line also carries a `secondary` block: the same measurement
(ms_per_step, tokens/s, gate_up fraction of the measured HBM bandwidth, layer
fraction, clocks) for every other headline configuration -- decode_c16 and
wide in W4A4, W4A16, MXFP4 and W4A8, decode_b512 in W4A4 and MXFP4 -- and the
single-expert GEMM sweep (FP4 TFLOPS at M=512 and the other M).
--no-secondary skips it.

--impl reference times the CPU oracle (the slow C restatement) on a bounded
sample of the same workload; it is the baseline arm, not a GPU code path.
Multi-GPU: the path does not shard (replicas only); every rank runs its own
replica and value = all ranks' tokens / max time.
"""
import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WEIGHT_BYTES_PER_ELEM = 0.5 + 1.0 / 16  # E2M1 codes + one E4M3 scale per 16
MX_WEIGHT_BYTES_PER_ELEM = 0.5 + 1.0 / 32  # MXFP4: E2M1 codes + one UE8M0 scale per 32


def _load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


def max_over_ranks(v, world, device="cpu"):
    """The largest value of v over the ranks of the job (the slowest replica
    sets the job's step time); v itself when there is one rank."""
    if world <= 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(units_per_rank, world, seconds_per_step):
    """Whole-job throughput: every rank processes its own units (replicas)."""
    return world * units_per_rank / seconds_per_step


def _dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled every 100 ms."""
    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.idx = gpu_index
        self.rows = []
        self.proc = None
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.idx), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return

        def reader():
            for line in self.proc.stdout:
                self.rows.append([c.strip() for c in line.split(",")])
        self.thread = threading.Thread(target=reader, daemon=True)
        self.thread.start()

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx = float(r[1])
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[4:8]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def _kernel_hash(mode="w4a4"):
    """Hash of the code of the dominant kernel of a mode (staleness check of
    the committed DRAM-traffic figure): its sources with comments and
    whitespace removed, so that only a change of code counts."""
    h = hashlib.sha256()
    src = {"w4a4": "gemm_w4a4.cu", "mxw4a4": "gemm_w4a4.cu", "w4a16": "gemm_w4a16.cu", "w4a8": "gemm_w4a16.cu"}[mode]
    for fn in (src, "common.cuh", "workitems.cuh"):
        with open(os.path.join(ROOT, "nvfp4_mixture_experts_top_gb300", "csrc", fn)) as f:
            src = f.read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)
        src = re.sub(r"//[^\n]*", " ", src)
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()[:16]


def _traffic(workload, mode):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary, or None if there is none or the kernel changed since."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get("%s/%s" % (workload, mode))
    if not e or e.get("kernel_hash") != _kernel_hash(mode):
        return None
    return e.get("dram_bytes_per_launch")


def gpu_weights(cfg, dev, B, wl, seed=0, mx=False):
    import torch
    if mx:
        return gpu_mx_weights(cfg, dev, B, wl, seed)
    out = []
    for which, N, K in (("w13", 2 * cfg.I, cfg.H), ("w2", cfg.H, cfg.I)):
        codes = torch.empty(cfg.E, N, K // 2, dtype=torch.uint8, device=dev)
        scales = torch.empty(cfg.E, N, K // 16, dtype=torch.uint8, device=dev)
        S = torch.empty(cfg.E, dtype=torch.float32, device=dev)
        for e in range(cfg.E):
            wf = wl.expert_weight_fp32(which, e, N, K, seed, device=dev)
            _, _, s = B.nvfp4_quantize(wf, codes=codes[e], scales=scales[e])
            S[e:e + 1].copy_(s)
        del wf
        packed = B.nvfp4_pack_weight_scales(scales, cfg.E, N, K)
        del scales
        out.append((codes, packed, S))
    return out


def gpu_mx_weights(cfg, dev, B, wl, seed=0):
    import torch
    out = []
    for which, N, K in (("w13", 2 * cfg.I, cfg.H), ("w2", cfg.H, cfg.I)):
        codes = torch.empty(cfg.E, N, K // 2, dtype=torch.uint8, device=dev)
        lin = torch.empty(cfg.E, N, K // 32, dtype=torch.uint8, device=dev)
        for e in range(cfg.E):
            wf = wl.expert_weight_fp32(which, e, N, K, seed, device=dev)
            _, s = B.mxfp4_quantize(wf, codes=codes[e])
            lin[e].copy_(s[:, : K // 32])
        del wf
        packed = B.mxfp4_pack_weight_scales(lin, cfg.E, N, K)
        del lin
        out.append((codes, packed, None))
    return out


def oracle_sample(cfg, mode, ntok, seed=0):
    """Prepare the oracle's inputs for the first `ntok` tokens of the
    workload (weights of the experts they use, quantised by the oracle; the
    whole batch's activation scale).  Returns a callable that runs the
    oracle's layer forward on that sample once."""
    from nvfp4_mixture_experts_top_gb300 import workloads as wl
    from oracle import oracle as orc
    x = wl.activations_bf16(cfg.T, cfg.H, seed).float().numpy()
    logits = wl.router_logits(cfg, seed).numpy()
    toks = list(range(ntok))
    ids, _ = orc.route(logits[toks], cfg.k)
    used = np.unique(ids)
    q = orc.mx_quantize_experts if mode == "mxw4a4" else orc.quantize_experts
    w13 = q(np.stack([wl.expert_weight_fp32("w13", e, 2 * cfg.I, cfg.H, seed).numpy() for e in used]))
    w2 = q(np.stack([wl.expert_weight_fp32("w2", e, cfg.H, cfg.I, seed).numpy() for e in used]))
    S_x = {"w4a4": orc.tensor_scale, "w4a8": orc.fp8_tensor_scale}[mode](x) if mode in ("w4a4", "w4a8") else None
    S_h = cfg.S_h8 if mode == "w4a8" else cfg.S_h
    xs, ls = x[toks], logits[toks][:, used]

    def run():
        orc.moe_layer(mode, xs, ls, cfg.k, w13, w2, S_h, S_x=S_x)
    return run


def cpu_baseline(cfg, mode, ntok, seconds=10.0, seed=0):
    """Time the oracle (as it stands) on the first `ntok` tokens of the
    workload on the host cores, repeating the sample until at least `seconds`
    of oracle work have run.  Returns (tokens/s, cores, seconds, passes)."""
    from oracle import oracle as orc
    ntok = min(ntok, cfg.T)
    run = oracle_sample(cfg, mode, ntok, seed)
    passes = 0
    t0 = time.perf_counter()
    while True:
        run()
        passes += 1
        dt = time.perf_counter() - t0
        if dt >= seconds:
            break
    return ntok * passes / dt, orc.num_threads(), dt, passes


def run_reference(args, cfg, metric, unit):
    ws, rank, _ = _dist()
    if rank != 0:
        return
    from oracle import oracle as orc
    ntok = args.ref_tokens
    run = oracle_sample(cfg, args.mode, ntok)
    times = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        run()
        if i >= args.warmup:
            times.append(time.perf_counter() - t0)
    ms = 1e3 * statistics.mean(times)
    val = ntok / (ms / 1e3)
    sample = "first %d tokens of the %s batch, oracle layer forward (weights pre-quantised)" % (ntok, cfg.name)
    line = {"impl": "reference", "metric": metric, "value": val, "unit": unit, "n_gpus": ws, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": cfg.name, "mode": args.mode, "T": cfg.T, "hidden": cfg.H,
                       "intermediate": cfg.I, "experts": cfg.E, "top_k": cfg.k, "routing": cfg.routing},
            "cpu_baseline": {"value": val, "unit": unit, "cores": orc.num_threads(), "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": val, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def gemm_sweep_rows(args, wl, Ms):
    """Single-expert NVFP4 GEMM, N=2048, K=6144, for each M in Ms: a CUDA
    graph of back-to-back GEMMs rotating over enough copies of A, W and out
    that their total exceeds twice the L2, so every launch reads its operands
    from HBM.  Returns (rows, fp4 peak TFLOP/s, peak kind)."""
    import torch

    from nvfp4_mixture_experts_top_gb300 import binding as B
    dev = torch.device("cuda", _dist()[2])
    torch.cuda.set_device(dev)
    B.load()
    B.nvfp4_device_check()
    hbm, bf16_tf, peak_kind = _load_peaks()
    fp4_peak = bf16_tf * 6.0  # nominal dense FP4 : BF16 ratio (13.5 / 2.25)
    N, K = wl.GEMM_SWEEP["N"], wl.GEMM_SWEEP["K"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    _, w = wl.gemm_operands_fp32(1, N, K, device=dev)
    wc, ws, wS = B.nvfp4_quantize(w)
    packed = B.nvfp4_pack_weight_scales(ws, 1, N, K)
    del w
    L = B.load()
    rows = []
    for M in Ms:
        a, _ = wl.gemm_operands_fp32(M, 1, K, device=dev)
        ac, as_, aS = B.nvfp4_quantize(a)
        del a
        per_copy = N * K * 0.5625 + M * K * 0.5625 + M * N * 4
        copies = int(max(2, np.ceil(2 * l2 / per_copy)))
        Ws = [(wc.clone(), packed.clone()) for _ in range(copies)]
        As = [(ac.clone(), as_.clone()) for _ in range(copies)]
        outs = [torch.empty(M, N, device=dev) for _ in range(copies)]
        offs = torch.tensor([0, M], dtype=torch.int32, device=dev)
        status = torch.zeros(1, dtype=torch.int32, device=dev)

        def launch(i):
            st = torch.cuda.current_stream().cuda_stream
            r = L.moe_grouped_gemm_nvfp4(0, As[i][0].data_ptr(), As[i][1].data_ptr(), aS.data_ptr(),
                                         Ws[i][0].data_ptr(), Ws[i][1].data_ptr(), wS.data_ptr(), offs.data_ptr(),
                                         1, N, K, M, outs[i].data_ptr(), status.data_ptr(), st)
            if r != 0:
                raise B.Nvfp4Error("moe_grouped_gemm_nvfp4", r)

        for i in range(args.warmup):
            launch(i % copies)
        reps = max(args.steps, copies)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(reps):
                    launch(i % copies)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError("device status %d" % int(status.item()))
        us = e0.elapsed_time(e1) * 1e3 / reps
        flops = 2.0 * M * N * K
        tflops = flops / (us * 1e-6) / 1e12
        gbs = per_copy / (us * 1e-6) / 1e9
        roof_us = max(per_copy / (hbm * 1e9), flops / (fp4_peak * 1e12)) * 1e6
        rows.append({"M": M, "us": us, "tflops": tflops, "gbs": gbs, "roofline_us": roof_us,
                     "frac_of_roofline": roof_us / us, "bound": "hbm" if per_copy / (hbm * 1e9) > flops / (
                         fp4_peak * 1e12) else "tensor", "copies": copies})
        del Ws, As, outs, g
    return rows, fp4_peak, peak_kind


def run_gemm_sweep(args, wl):
    """The GEMM sweep as the benchmark's line: value = FP4 TFLOPS at M=512."""
    Ms = [int(m) for m in args.sweep_ms.split(",")] if args.sweep_ms else list(wl.GEMM_SWEEP["Ms"])
    N, K = wl.GEMM_SWEEP["N"], wl.GEMM_SWEEP["K"]
    rows, fp4_peak, peak_kind = gemm_sweep_rows(args, wl, Ms)
    m512 = ([r for r in rows if r["M"] == 512] or rows)[0]
    result = {"metric": "FP4 TFLOPS at M=%d (single-expert NVFP4 GEMM, N=2048, K=6144)" % m512["M"],
              "value": m512["tflops"],
              "unit": "TFLOP/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
              "ms_per_step": m512["us"] / 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
              "dtype": "fp4(e2m1)xfp4, fp32 accumulate", "data": "synthetic",
              "config": {"workload": "gemm_sweep", "N": N, "K": K, "Ms": Ms,
                         "l2": "rotating %d+ operand copies > 2x L2" % min(r["copies"] for r in rows)},
              "roofline": {"bound": m512["bound"], "achieved": m512["tflops"], "peak": fp4_peak, "unit": "TFLOP/s",
                           "frac": m512["tflops"] / fp4_peak,
                           "peak_kind": "measured bf16 x nominal fp4/bf16 ratio 6 (%s)" % peak_kind,
                           "traffic": None},
              "sweep": rows, "gpu_launches": 1}
    print(json.dumps(result), flush=True)


def run_router(args, cfg, wl):
    """Router for the workload's T, H, E, k: graphs of back-to-back calls
    rotating over copies of x and W_router whose total exceeds twice the L2,
    so every call reads its operands from HBM.  Three forms are timed:
    moe_router_logits alone; moe_router_logits + moe_align_permute (the
    staged router and routing); moe_router_route (router and routing in one
    call: the router GEMM and, for T <= 32, one fused reduce/top-k/permute
    kernel).  value = tokens/s of moe_router_route."""
    import torch

    from nvfp4_mixture_experts_top_gb300 import binding as B
    dev = torch.device("cuda", _dist()[2])
    torch.cuda.set_device(dev)
    L = B.load()
    B.nvfp4_device_check()
    hbm, _, peak_kind = _load_peaks()
    T, H, E, k = cfg.T, cfg.H, cfg.E, cfg.k
    R = T * k
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    per_copy = E * H * 2 + T * H * 2 + T * E * 4
    copies = int(max(2, np.ceil(2 * l2 / per_copy)))
    x = wl.activations_bf16(T, H, device=dev)
    w = wl.router_weight_bf16(E, H, device=dev)
    Xs = [x.clone() for _ in range(copies)]
    Ws = [w.clone() for _ in range(copies)]
    outs = [torch.empty(T, E, device=dev) for _ in range(copies)]
    ws = torch.empty(int(L.moe_router_logits_workspace_bytes(T, H, E)), dtype=torch.uint8, device=dev)
    ws_rr = torch.empty(int(L.moe_router_route_workspace_bytes(T, H, E, k)), dtype=torch.uint8, device=dev)
    ws_rt = torch.empty(max(int(L.moe_align_permute_workspace_bytes(T, E, k)), 256), dtype=torch.uint8, device=dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, k, dtype=torch.float32, device=dev)
    offs = torch.empty(E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(R, dtype=torch.int32, device=dev)
    inv = torch.empty(R, dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    P = lambda t: None if t is None else t.data_ptr()  # noqa: E731

    def chk(name, r):
        if r != 0:
            raise B.Nvfp4Error(name, r)

    def logits_only(i):
        chk("moe_router_logits", L.moe_router_logits(P(Xs[i]), P(Ws[i]), T, H, E, P(outs[i]), P(status), P(ws),
                                                      ws.numel(), torch.cuda.current_stream().cuda_stream))

    def staged(i):
        logits_only(i)
        chk("moe_align_permute", L.moe_align_permute(P(outs[i]), T, E, k, P(ids), P(tw), P(offs), P(perm), P(inv), 0,
                                                      None, None, 0, None, None, P(status), P(ws_rt), ws_rt.numel(),
                                                      torch.cuda.current_stream().cuda_stream))

    def fused(i):
        chk("moe_router_route", L.moe_router_route(P(Xs[i]), P(Ws[i]), T, H, E, k, P(outs[i]), P(ids), P(tw),
                                                    P(offs), P(perm), P(inv), P(status), P(ws_rr), ws_rr.numel(),
                                                    torch.cuda.current_stream().cuda_stream))

    def time_graph(fn):
        for i in range(args.warmup):
            fn(i % copies)
        reps = max(args.steps, copies)
        side = torch.cuda.Stream()
        side.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(g, stream=side):
                for i in range(reps):
                    fn(i % copies)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record()
        g.replay()
        e1.record()
        torch.cuda.synchronize()
        if int(status.item()) != 0:
            raise RuntimeError("device status %d" % int(status.item()))
        return e0.elapsed_time(e1) * 1e3 / reps, reps

    us_logits, _ = time_graph(logits_only)
    us_staged, _ = time_graph(staged)
    us, reps = time_graph(fused)
    gbs = per_copy / (us_logits * 1e-6) / 1e9
    splits = int(L.moe_router_logits_workspace_bytes(T, H, E)) // max(1, T * E * 4)
    fused_kernels = 2 if T <= 32 else (3 if splits > 1 else 2)
    result = {"metric": "router + routing tokens/s (%s: T=%d, H=%d, E=%d, top-%d)" % (cfg.name, T, H, E, k),
              "value": T / (us * 1e-6), "unit": "tokens/s", "n_gpus": 1, "steps": reps, "warmup": args.warmup,
              "ms_per_step": us / 1e3, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
              "dtype": "bf16xbf16, fp32 accumulate", "data": "synthetic",
              "config": {"workload": cfg.name + "_router", "T": T, "hidden": H, "experts": E, "top_k": k,
                         "k_splits": max(1, splits), "l2": "rotating %d operand copies > 2x L2" % copies},
              "router_logits_us": us_logits, "router_then_align_permute_us": us_staged, "router_route_us": us,
              "roofline": {"kernel": "router logits GEMM (+ reduce)", "bound": "hbm", "achieved": gbs, "peak": hbm,
                           "unit": "GB/s", "frac": gbs / hbm, "peak_kind": peak_kind,
                           "algorithmic_bytes_per_launch": per_copy, "avg_launch_us": us_logits, "traffic": None},
              "gpu_launches": reps * fused_kernels}
    print(json.dumps(result), flush=True)


def measure_layer(args, cfg, mode_name, metric, world, rank, local, full=True, no_clocks=False):
    """Time the layer of one workload and mode (see the module docstring);
    full=True adds the end-to-end host-buffer measurement.  Returns the
    result dict of the JSON line (without cpu_baseline)."""
    import torch
    import torch.distributed as dist

    from nvfp4_mixture_experts_top_gb300 import binding as B
    from nvfp4_mixture_experts_top_gb300 import workloads as wl
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mode = {"w4a4": B.MOE_W4A4, "w4a16": B.MOE_W4A16, "mxw4a4": B.MOE_MXW4A4, "w4a8": B.MOE_W4A8}[mode_name]
    mx = mode == B.MOE_MXW4A4
    bpe = MX_WEIGHT_BYTES_PER_ELEM if mx else WEIGHT_BYTES_PER_ELEM

    (w13, w2) = gpu_weights(cfg, dev, B, wl, mx=mx)
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    logits = wl.router_logits(cfg, device=dev)
    S_h = torch.tensor([cfg.S_h8 if mode == B.MOE_W4A8 else cfg.S_h], dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    I, H, k, T, R = cfg.I, cfg.H, cfg.k, cfg.T, cfg.R

    # intermediates of the staged step (same kernels as moe_layer_forward)
    ws_route = torch.empty(max(B.load().moe_align_permute_workspace_bytes(T, cfg.E, k), 256), dtype=torch.uint8,
                           device=dev)
    S_x = torch.zeros(4, dtype=torch.float32, device=dev)
    ids = torch.empty(T, k, dtype=torch.int32, device=dev)
    tw = torch.empty(T, k, dtype=torch.float32, device=dev)
    offs = torch.empty(cfg.E + 1, dtype=torch.int32, device=dev)
    perm = torch.empty(R, dtype=torch.int32, device=dev)
    inv = torch.empty(R, dtype=torch.int32, device=dev)
    a_c = torch.empty(R, H if mode == B.MOE_W4A8 else H // 2, dtype=torch.uint8, device=dev)
    a_s = torch.empty(R, B.mxfp4_scale_pitch(H) if mx else H // 16, dtype=torch.uint8, device=dev)
    a_b = torch.empty(R, H, dtype=torch.bfloat16, device=dev)
    G = torch.empty(R, 2 * I, dtype=torch.float32, device=dev)
    h_c = torch.empty(R, I if mode == B.MOE_W4A8 else I // 2, dtype=torch.uint8, device=dev)
    h_s = torch.empty(R, B.mxfp4_scale_pitch(I) if mx else I // 16, dtype=torch.uint8, device=dev)
    h_b = torch.empty(R, I, dtype=torch.bfloat16, device=dev)
    a_rs = torch.empty(R, dtype=torch.float32, device=dev)  # W4A16: F16 row carriers' multipliers
    h_rs = torch.empty(R, dtype=torch.float32, device=dev)
    Y = torch.empty(R, H, dtype=torch.float32, device=dev)
    out = torch.empty(T, H, dtype=torch.float32, device=dev)
    L = B.load()
    P = lambda t: None if t is None else t.data_ptr()  # noqa: E731

    def chk(s):
        if s != 0:
            raise B.Nvfp4Error("step", s)

    def step(ev_pair=None):
        st = torch.cuda.current_stream().cuda_stream
        if mx:
            # routing + MXFP4 quantisation straight into permuted rows
            chk(L.moe_route_quantize_mxfp4(P(x), P(logits), T, H, cfg.E, k, P(ids), P(tw), P(offs), P(perm),
                                           P(inv), P(a_c), P(a_s), P(status), P(ws_route), ws_route.numel(), st))
            if ev_pair:
                ev_pair[0].record()
            chk(L.moe_grouped_gemm_nvfp4(2, P(a_c), P(a_s), None, P(w13[0]), P(w13[1]), None, P(offs),
                                         cfg.E, 2 * I, H, R, P(G), P(status), st))
            if ev_pair:
                ev_pair[1].record()
            chk(L.moe_swiglu_requant(P(G), R, I, 2, None, P(h_c), P(h_s), None, st))
            chk(L.moe_grouped_gemm_nvfp4(2, P(h_c), P(h_s), None, P(w2[0]), P(w2[1]), None, P(offs),
                                         cfg.E, H, I, R, P(Y), P(status), st))
        elif mode == B.MOE_W4A8:
            # as moe_layer_forward runs it: routing + FP8 quantisation straight
            # into permuted rows, the codes carried as their f16 values into
            # the F16-operand GEMM (MOE_W4A16F)
            chk(L.moe_route_quantize_fp8_f16(P(x), P(logits), T, H, cfg.E, k, P(ids), P(tw), P(offs), P(perm),
                                             P(inv), P(S_x), P(a_b), P(a_rs), P(status), P(ws_route),
                                             ws_route.numel(), st))
            if ev_pair:
                ev_pair[0].record()
            chk(L.moe_grouped_gemm_nvfp4(4, P(a_b), None, P(a_rs), P(w13[0]), P(w13[1]), P(w13[2]), P(offs),
                                         cfg.E, 2 * I, H, R, P(G), P(status), st))
            if ev_pair:
                ev_pair[1].record()
            chk(L.moe_swiglu_fp8_f16(P(G), R, I, P(S_h), P(h_b), P(h_rs), st))
            chk(L.moe_grouped_gemm_nvfp4(4, P(h_b), None, P(h_rs), P(w2[0]), P(w2[1]), P(w2[2]), P(offs),
                                         cfg.E, H, I, R, P(Y), P(status), st))
        elif mode == B.MOE_W4A4:
            # routing + activation quantisation straight into permuted rows
            # (the kernels moe_layer_forward runs)
            chk(L.moe_route_quantize_nvfp4(P(x), P(logits), T, H, cfg.E, k, P(ids), P(tw), P(offs), P(perm),
                                           P(inv), P(S_x), P(a_c), P(a_s), P(status), P(ws_route),
                                           ws_route.numel(), st))
            if ev_pair:
                ev_pair[0].record()
            chk(L.moe_grouped_gemm_nvfp4(0, P(a_c), P(a_s), P(S_x), P(w13[0]), P(w13[1]), P(w13[2]), P(offs),
                                         cfg.E, 2 * I, H, R, P(G), P(status), st))
            if ev_pair:
                ev_pair[1].record()
            chk(L.moe_swiglu_requant(P(G), R, I, 0, P(S_h), P(h_c), P(h_s), None, st))
            chk(L.moe_grouped_gemm_nvfp4(0, P(h_c), P(h_s), P(S_h), P(w2[0]), P(w2[1]), P(w2[2]), P(offs),
                                         cfg.E, H, I, R, P(Y), P(status), st))
        else:
            # W4A16 as moe_layer_forward runs it: the bf16 operands carried as
            # F16 rows with per-row powers of two (GEMM mode MOE_W4A16F)
            chk(L.moe_align_permute(P(logits), T, cfg.E, k, P(ids), P(tw), P(offs), P(perm), P(inv), 0, None, None,
                                    0, None, None, P(status), P(ws_route), ws_route.numel(), st))
            chk(L.moe_gather_f16(P(x), T, H, P(perm), R, P(a_b), P(a_rs), st))
            if ev_pair:
                ev_pair[0].record()
            chk(L.moe_grouped_gemm_nvfp4(4, P(a_b), None, P(a_rs), P(w13[0]), P(w13[1]), P(w13[2]), P(offs),
                                         cfg.E, 2 * I, H, R, P(G), P(status), st))
            if ev_pair:
                ev_pair[1].record()
            chk(L.moe_swiglu_f16(P(G), R, I, P(h_b), P(h_rs), st))
            chk(L.moe_grouped_gemm_nvfp4(4, P(h_b), None, P(h_rs), P(w2[0]), P(w2[1]), P(w2[2]), P(offs),
                                         cfg.E, H, I, R, P(Y), P(status), st))
        chk(L.moe_combine(P(Y), P(inv), P(tw), T, k, H, 1, P(out), P(status), st))

    # kernels of this library per step: W4A4 route, quantise-scatter, 2 GEMMs,
    # SwiGLU-requant, combine; W4A16 route, gather, 2 GEMMs, SwiGLU, combine
    launches_per_step = 6

    # warm-up (eager)
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if int(status.item()) != 0:
        raise RuntimeError("device status %d after warm-up" % int(status.item()))
    # the staged step and the one-call layer agree bit for bit
    layer_out = torch.empty(T, H, dtype=torch.float32, device=dev)
    layer_ws = torch.empty(B.moe_layer_workspace_bytes(mode, T, H, I, cfg.E, k), dtype=torch.uint8, device=dev)

    def layer_step():
        B.moe_layer_forward(mode, x, logits, k, w13, w2, S_h, out=layer_out, workspace=layer_ws, dev_status=status)

    for _ in range(args.warmup):
        layer_step()
    torch.cuda.synchronize()
    if not torch.equal(layer_out, out):
        raise RuntimeError("staged step and moe_layer_forward disagree")

    # touched experts -> algorithmic bytes
    counts = np.diff(offs.cpu().numpy())
    touched = int((counts > 0).sum())
    w13_bytes = touched * 2 * I * H * bpe
    w2_bytes = touched * H * I * bpe
    act_in = R * H * {B.MOE_W4A16: 2.0, B.MOE_W4A8: 2.0}.get(mode, bpe)  # both carried as f16 rows
    gemm1_bytes = w13_bytes + act_in + R * 2 * I * 4
    layer_weight_bytes = w13_bytes + w2_bytes

    # two graphs of K steps: the layer as a user runs it (K moe_layer_forward
    # calls: kernels back to back, each a programmatic dependent of the one
    # before), and the staged entry points with event nodes around every
    # gate_up GEMM for its own duration (an event node between two kernels
    # makes the second wait for the first's end)
    K = args.steps
    def timing_event():
        # recorded inside the captured graph: must be an external event node
        return torch.cuda.Event(enable_timing=True, external=True)

    evs = [(timing_event(), timing_event()) for _ in range(K)]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    graph_ev = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            for i in range(K):
                layer_step()
        with torch.cuda.graph(graph_ev, stream=side):
            for i in range(K):
                step(evs[i])
    torch.cuda.synchronize()
    graph.replay()  # one untimed replay of each (graph upload)
    graph_ev.replay()
    torch.cuda.synchronize()

    clocks = ClockSampler(local)
    if not no_clocks:
        clocks.start()
        t_end = time.time() + 1.0  # clock window under load before the timed region
        while time.time() < t_end:
            graph.replay()
        torch.cuda.synchronize()

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    # profiler range = the timed region (ncu --profile-from-start off)
    torch.cuda.profiler.start()
    t0.record()
    graph.replay()
    t1.record()
    torch.cuda.synchronize()
    torch.cuda.profiler.stop()
    graph_ev.replay()  # the gate_up GEMM durations (second timed pass)
    torch.cuda.synchronize()
    # spread: five more replays of the layer graph after the timed one
    spread = [ms_total_timed := t0.elapsed_time(t1)]
    for _ in range(5):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        graph.replay()
        b.record()
        torch.cuda.synchronize()
        spread.append(a.elapsed_time(b))
    spread = sorted(v / K for v in spread)
    if world > 1:
        dist.barrier()
    if not no_clocks:
        clocks.stop()
    ms_total = ms_total_timed
    gemm_ms = [a.elapsed_time(b) for a, b in evs]
    if int(status.item()) != 0:
        raise RuntimeError("device status %d" % int(status.item()))
    if not torch.equal(layer_out, out):
        raise RuntimeError("timed layer output differs from the staged step")
    ms_step = max_over_ranks(ms_total / K, world, dev)
    value = job_throughput(T, world, ms_step / 1e3)

    e2e = None
    if full:
        # end to end through the public API with host buffers: MoELayerGraph
        # replays moe_layer_forward_host (inputs read from and output written
        # to pinned host memory by the layer's own kernels) as one graph; each
        # step also waits for the result on the host
        lg_graph = B.MoELayerGraph(mode, T, H, cfg.E, k, w13, w2, S_h, device=dev)
        lg_graph.x_host.copy_(x.cpu())
        lg_graph.logits_host.copy_(logits.cpu())
        for _ in range(args.warmup):
            lg_graph.run()
        te0 = time.perf_counter()
        for _ in range(K):
            res = lg_graph.run()
        e2e_s = max_over_ranks((time.perf_counter() - te0) / K, world, dev)
        if not torch.equal(res, out.cpu()):
            raise RuntimeError("e2e result differs from the device-timed step")
        if int(lg_graph.dev_status.item()) != 0:
            raise RuntimeError("device status %d in the e2e run" % int(lg_graph.dev_status.item()))
        e2e = {"value": job_throughput(T, world, e2e_s), "unit": "tokens/s",
               "h2d_bytes_per_step": x.numel() * 2 + logits.numel() * 4, "d2h_bytes_per_step": out.numel() * 4}
        del lg_graph

    hbm, _, peak_kind = _load_peaks()
    gemm_avg_ms = statistics.mean(gemm_ms)
    achieved = gemm1_bytes / (gemm_avg_ms / 1e3) / 1e9
    result = {
        "metric": metric, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": ms_step, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": {B.MOE_W4A4: "fp4(e2m1)xfp4, fp32 accumulate", B.MOE_W4A16: "fp4(e2m1)xbf16 (carried as f16 rows), fp32 accumulate",
                  B.MOE_MXW4A4: "fp4(e2m1)xfp4 (UE8M0 scales), fp32 accumulate",
                  B.MOE_W4A8: "fp4(e2m1)xfp8(e4m3) (codes carried as f16 values), fp32 accumulate"}[mode],
        "data": "synthetic (seeded N(0,1) bf16 activations, N(0,0.02) weights quantised on the GPU)",
        "config": {"workload": cfg.name, "mode": mode_name, "T": T, "hidden": H, "intermediate": I,
                   "experts": cfg.E, "top_k": k, "routing": cfg.routing, "touched_experts": touched,
                   "parallelism": "replicas" if world > 1 else "single GPU",
                   "l2": "no flush: %.2f GB of touched weights per step >> 129 MB L2" % (layer_weight_bytes / 1e9),
                   "timing": "CUDA graph of %d moe_layer_forward calls, CUDA events; gate_up duration from a "
                             "second graph of the %d steps through the staged entry points with events around "
                             "each gate_up launch" % (K, K)},
        "roofline": {"kernel": "moe_grouped_gemm_nvfp4 gate_up (%s)" % mode_name, "bound": "hbm",
                     "achieved": achieved, "peak": hbm, "unit": "GB/s", "frac": achieved / hbm,
                     "peak_kind": peak_kind, "algorithmic_bytes_per_launch": gemm1_bytes,
                     "avg_launch_ms": gemm_avg_ms, "traffic": _traffic(cfg.name, mode_name)},
        "layer_hbm": {"weight_bytes_per_step": layer_weight_bytes,
                      "achieved_gbs": layer_weight_bytes / (ms_step / 1e3) / 1e9,
                      "frac_of_peak": layer_weight_bytes / (ms_step / 1e3) / 1e9 / hbm},
        "e2e": e2e,
        "gpu_launches": launches_per_step * K,
        "spread": {"replays": len(spread), "ms_per_step_min": spread[0],
                   "ms_per_step_median": statistics.median(spread), "ms_per_step_max": spread[-1],
                   "note": "the timed replay and five more of the same graph"},
    }
    if not no_clocks:
        result["clocks"] = clocks.summary()
    return result


def layer_metric(cfg, mode_name):
    if mode_name == "mxw4a4":
        return "MoE-layer tokens/s (MXFP4 W4A4, %s)" % cfg.name
    if mode_name == "w4a8":
        return "MoE-layer tokens/s (NVFP4 weights, FP8 activations, %s)" % cfg.name
    return "MoE-layer tokens/s (NVFP4 %s, %s)" % (mode_name.upper(), cfg.name)


# The headline configurations other than the one the line is quoted on; the
# default run measures each of them too (secondary block of the line).
SECONDARY = (("decode_c16", "w4a16"), ("decode_c16", "mxw4a4"), ("decode_c16", "w4a8"), ("decode_b512", "w4a4"),
             ("decode_b512", "mxw4a4"), ("wide", "w4a4"), ("wide", "w4a16"), ("wide", "mxw4a4"), ("wide", "w4a8"))


def secondary_entry(r):
    """The compact form of a measure_layer() result for the secondary block."""
    return {"metric": r["metric"], "value": r["value"], "unit": r["unit"], "ms_per_step": r["ms_per_step"],
            "config": r["config"], "frac": r["roofline"]["frac"], "gate_up_ms": r["roofline"]["avg_launch_ms"],
            "layer_frac": r["layer_hbm"]["frac_of_peak"], "clocks": r.get("clocks"),
            "spread": r["spread"]}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="decode_c16",
                    choices=["decode_c16", "decode_b512", "wide", "tiny", "gemm_sweep"])
    ap.add_argument("--mode", default="w4a4", choices=["w4a4", "w4a16", "mxw4a4", "w4a8"])
    ap.add_argument("--ref-tokens", type=int, default=1, help="tokens per reference-arm step")
    ap.add_argument("--baseline-tokens", type=int, default=16, help="tokens of the in-run CPU baseline sample")
    ap.add_argument("--baseline-seconds", type=float, default=10.0,
                    help="the in-run CPU baseline repeats its sample for at least this long")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-clocks", action="store_true")
    ap.add_argument("--no-secondary", action="store_true",
                    help="measure only the selected workload (no secondary block of the other headline configs)")
    ap.add_argument("--router", action="store_true",
                    help="time the router-logits GEMM for the workload's T, H, E instead of the layer")
    ap.add_argument("--sweep-ms", default="",
                    help="gemm_sweep: comma-separated subset of the M values (e.g. for a profiler capture)")
    ap.add_argument("--experts", type=int, default=0,
                    help="override the expert count (smaller device footprint for profiler captures)")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    from nvfp4_mixture_experts_top_gb300 import workloads as wl
    if args.workload == "gemm_sweep":
        return run_gemm_sweep(args, wl)
    cfg = wl.CONFIGS[args.workload]
    if args.experts:
        cfg = wl.small_variant(cfg, E=args.experts, name=cfg.name + "_E%d" % args.experts)
    if args.router:
        return run_router(args, cfg, wl)
    metric = layer_metric(cfg, args.mode)
    unit = "tokens/s"
    if args.impl == "reference":
        return run_reference(args, cfg, metric, unit)

    import torch
    import torch.distributed as dist

    from nvfp4_mixture_experts_top_gb300 import binding as B
    world, rank, local = _dist()
    if world > 1:
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    B.load()
    B.nvfp4_device_check()
    result = measure_layer(args, cfg, args.mode, metric, world, rank, local, full=True, no_clocks=args.no_clocks)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        v, cores, dt, passes = cpu_baseline(cfg, args.mode, args.baseline_tokens, args.baseline_seconds)
        result["cpu_baseline"] = {"value": v, "unit": unit, "cores": cores, "kind": "oracle",
                                  "sample": "first %d tokens of the batch, oracle layer forward %d times "
                                            "(%.1f s of oracle work)" % (min(args.baseline_tokens, cfg.T),
                                                                         passes, dt)}
    if world == 1 and not args.no_secondary and not args.experts:
        # every other headline configuration, each measured the same way
        sec = []
        for wname, mname in SECONDARY:
            if (wname, mname) == (cfg.name, args.mode):
                continue
            c2 = wl.CONFIGS[wname]
            r2 = measure_layer(args, c2, mname, layer_metric(c2, mname), world, rank, local, full=False,
                               no_clocks=args.no_clocks)
            sec.append(secondary_entry(r2))
            torch.cuda.empty_cache()
        if (cfg.name, args.mode) != ("decode_c16", "w4a4"):
            r2 = measure_layer(args, wl.CONFIGS["decode_c16"], "w4a4", layer_metric(wl.CONFIGS["decode_c16"], "w4a4"),
                               world, rank, local, full=False, no_clocks=args.no_clocks)
            sec.insert(0, secondary_entry(r2))
        # the single-expert GEMM sweep: FP4 TFLOPS at M=512 (and the other M)
        rows, fp4_peak, peak_kind = gemm_sweep_rows(args, wl, list(wl.GEMM_SWEEP["Ms"]))
        m512 = [r for r in rows if r["M"] == 512][0]
        sec.append({"metric": "FP4 TFLOPS at M=512 (single-expert NVFP4 GEMM, N=2048, K=6144)",
                    "value": m512["tflops"], "unit": "TFLOP/s", "ms_per_step": m512["us"] / 1e3,
                    "config": {"workload": "gemm_sweep", "N": wl.GEMM_SWEEP["N"], "K": wl.GEMM_SWEEP["K"],
                               "Ms": list(wl.GEMM_SWEEP["Ms"])},
                    "frac": m512["tflops"] / fp4_peak,
                    "peak": fp4_peak, "peak_kind": "measured bf16 x nominal fp4/bf16 ratio 6 (%s)" % peak_kind,
                    "frac_of_roofline": m512["frac_of_roofline"], "sweep": rows})
        result["secondary"] = sec
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
