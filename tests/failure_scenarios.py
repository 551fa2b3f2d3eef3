"""Failure-detection scenarios, each run in a child process by
test_gpu_failure.py.

The library reads NVFP4MOE_TEST_DROP_STAGE=n once per process and applies it
to the first grouped-GEMM or router-GEMM launch only: that launch never arms
its pipeline stage n, so its bounded waits run out.  A scenario therefore runs
in a fresh process with the variable set.  It makes the injected call, which
must report NVFP4_E_DEVICE_TIMEOUT in the status word and return (no trap, no
hang), and then repeats the call in the same process and CUDA context, which
must give the oracle's result with a clean status.

    python failure_scenarios.py <scenario> [mode]

prints one JSON line with the two statuses, the injected call's wall time and
the error of the repeated call; the exit status is nonzero if a check fails.
"""
import json
import os
import sys
import time

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from gpu_helpers import assert_close, to_dev, upload_weights  # noqa: E402
from nvfp4_mixture_experts_top_gb300 import binding as B  # noqa: E402
from nvfp4_mixture_experts_top_gb300 import workloads as wl  # noqa: E402
from oracle import oracle as orc  # noqa: E402

NVFP4_E_DEVICE_TIMEOUT = 7


def _timed(fn):
    t0 = time.time()
    fn()
    torch.cuda.synchronize()
    return time.time() - t0


def gemm(dev, mode):
    E, N, K = 2, 128, 512
    offs = np.array([0, 5, 8], np.int32)
    if mode == "w4a4":
        w = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w13", e, N, K).numpy() for e in range(E)]))
        a = wl.random_fp32((8, K), seed=1, tag="fail").to(torch.bfloat16).float().numpy()
        ac, as_, aS = orc.quantize(a)
        args = (to_dev(ac, dev), to_dev(as_, dev), to_dev(np.array([aS]), dev), *upload_weights(w, E, N, K, dev),
                to_dev(offs, dev), N, K)
        m = B.MOE_W4A4
        ref = lambda: orc.grouped_gemm_w4a4(ac, as_, aS, w[0], w[1], w[2], offs)  # noqa: E731
    elif mode == "w4a8":
        w = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w2", e, N, K).numpy() for e in range(E)]))
        a = wl.random_fp32((8, K), seed=3, tag="fail8").to(torch.bfloat16).float().numpy()
        ac, aS = orc.fp8_quantize(a)
        args = (to_dev(ac, dev), None, to_dev(np.array([aS]), dev), *upload_weights(w, E, N, K, dev),
                to_dev(offs, dev), N, K)
        m = B.MOE_W4A8
        ref = lambda: orc.grouped_gemm_w4a8(ac, aS, w[0], w[1], w[2], offs)  # noqa: E731
    else:
        w = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w2", e, N, K).numpy() for e in range(E)]))
        a = wl.random_fp32((8, K), seed=2, tag="fail16").to(torch.bfloat16).float().numpy()
        args = (to_dev(a, dev, torch.bfloat16), None, None, *upload_weights(w, E, N, K, dev), to_dev(offs, dev), N, K)
        m = B.MOE_W4A16
        ref = lambda: orc.grouped_gemm_w4a16(a, w[0], w[1], w[2], offs)  # noqa: E731
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    elapsed = _timed(lambda: B.moe_grouped_gemm_nvfp4(m, *args, dev_status=status))
    first = int(status.item())
    status.zero_()
    out = B.moe_grouped_gemm_nvfp4(m, *args, dev_status=status)
    torch.cuda.synchronize()
    return first, int(status.item()), elapsed, out.cpu().numpy(), ref()


def gemm_pair(dev, mode):
    """The CTA-pair GEMM (many tokens per expert): both CTAs of a pair skip
    the same stage, so both sides' bounded waits run out."""
    E, N, K = 1, 256, 1024
    offs = np.array([0, 1024], np.int32)
    w = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w13", 0, N, K, 6).numpy()]))
    a = wl.random_fp32((1024, K), seed=6, tag="failpair").to(torch.bfloat16).float().numpy()
    ac, as_, aS = orc.quantize(a)
    args = (to_dev(ac, dev), to_dev(as_, dev), to_dev(np.array([aS]), dev), *upload_weights(w, E, N, K, dev),
            to_dev(offs, dev), N, K)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    elapsed = _timed(lambda: B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, *args, dev_status=status))
    first = int(status.item())
    status.zero_()
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, *args, dev_status=status)
    torch.cuda.synchronize()
    return first, int(status.item()), elapsed, out.cpu().numpy(), orc.grouped_gemm_w4a4(ac, as_, aS, w[0], w[1],
                                                                                          w[2], offs)


def router(dev, mode):
    T, H, E = 16, 1024, 256
    x = wl.activations_bf16(T, H, seed=4)
    wr = wl.router_weight_bf16(E, H, seed=4)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    elapsed = _timed(lambda: B.moe_router_logits(x.to(dev), wr.to(dev), dev_status=status))
    first = int(status.item())
    status.zero_()
    got = B.moe_router_logits(x.to(dev), wr.to(dev), dev_status=status)
    torch.cuda.synchronize()
    return first, int(status.item()), elapsed, got.cpu().numpy(), orc.router_logits(x.float().numpy(),
                                                                                      wr.float().numpy())


def layer(dev, mode):
    """The whole layer, its kernels chained as programmatic dependents: the
    injected gate_up GEMM times out, the kernels after it still run and
    return, and the next layer call is correct.  H = 4096 gives at least four
    K stages per gate_up work unit after the K split (16 stages in up to four
    parts), so stage 3 lies inside the first ring lap."""
    cfg = wl.MoEConfig("fail_layer", T=8, H=4096, I=512, E=4, k=2, routing="uniform")
    m = {"w4a4": B.MOE_W4A4, "w4a16": B.MOE_W4A16}[mode]
    xt = wl.activations_bf16(cfg.T, cfg.H, seed=5)
    logits = wl.router_logits(cfg, seed=5)
    w13 = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w13", e, 2 * cfg.I, cfg.H, 5).numpy()
                                         for e in range(cfg.E)]))
    w2 = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w2", e, cfg.H, cfg.I, 5).numpy()
                                        for e in range(cfg.E)]))
    g13 = upload_weights(w13, cfg.E, 2 * cfg.I, cfg.H, dev)
    g2 = upload_weights(w2, cfg.E, cfg.H, cfg.I, dev)
    S_h = torch.tensor([cfg.S_h], dtype=torch.float32, device=dev)
    x, lg = xt.to(dev), logits.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    elapsed = _timed(lambda: B.moe_layer_forward(m, x, lg, cfg.k, g13, g2, S_h, dev_status=status))
    first = int(status.item())
    status.zero_()
    out = B.moe_layer_forward(m, x, lg, cfg.k, g13, g2, S_h, dev_status=status)
    torch.cuda.synchronize()
    ref = orc.moe_layer(mode, xt.float().numpy(), logits.numpy(), cfg.k, w13, w2, cfg.S_h)
    return first, int(status.item()), elapsed, out.cpu().numpy(), ref


SCENARIOS = {"gemm": gemm, "gemm_pair": gemm_pair, "router": router, "layer": layer}


def main():
    name = sys.argv[1]
    mode = sys.argv[2] if len(sys.argv) > 2 else "w4a4"
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    B.load(build_if_missing=False)
    B.nvfp4_device_check()
    orc.lib()
    first, after, elapsed, got, ref = SCENARIOS[name](dev, mode)
    rel, mx = assert_close(got, ref, "%s %s after the timeout" % (name, mode))
    print(json.dumps({"scenario": name, "mode": mode, "drop": os.environ.get("NVFP4MOE_TEST_DROP_STAGE"),
                      "status_injected": first, "status_after": after, "elapsed_s": elapsed,
                      "rel_frob": rel, "max_over_rms": mx}))
    ok = first == NVFP4_E_DEVICE_TIMEOUT and after == 0 and elapsed < 30.0
    sys.exit(0 if ok else 1)


if __name__ == "__main__":
    main()
