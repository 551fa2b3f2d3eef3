"""Failure detection on the GPU without faulting it.

The grouped GEMMs' (W4A4 and W4A16) and the router GEMM's waits are bounded.  With the test-only fault injection
(NVFP4MOE_TEST_DROP_STAGE: the producer never arms one pipeline stage) the
consumers' waits run out: the kernel must report NVFP4_E_DEVICE_TIMEOUT in
the status word, drain its copies and MMAs, free its tensor memory and
return -- and the context must stay usable: the same GEMM right after gives
the oracle's result.  Routing errors are reported the same way (status word,
no trap): see test_gpu_gemm.py::test_gemm_bad_offsets_report_status.
"""
import os
import time

import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev, upload_weights
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

NVFP4_E_DEVICE_TIMEOUT = 7


def test_gemm_bounded_wait_times_out_and_context_survives(orc):
    dev = cuda_or_skip()
    E, N, K = 2, 128, 512
    counts = [5, 3]
    offs = np.array([0, 5, 8], np.int32)
    w = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w13", e, N, K).numpy() for e in range(E)]))
    a = wl.random_fp32((8, K), seed=1, tag="fail").to(torch.bfloat16).float().numpy()
    ac, as_, aS = orc.quantize(a)
    wd = upload_weights(w, E, N, K, dev)
    args = (to_dev(ac, dev), to_dev(as_, dev), to_dev(np.array([aS]), dev), *wd, to_dev(offs, dev), N, K)

    status = torch.zeros(1, dtype=torch.int32, device=dev)
    os.environ["NVFP4MOE_TEST_DROP_STAGE"] = "0"
    try:
        t0 = time.time()
        B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, *args, dev_status=status)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        del os.environ["NVFP4MOE_TEST_DROP_STAGE"]
    assert int(status.item()) == NVFP4_E_DEVICE_TIMEOUT
    assert elapsed < 30.0

    status.zero_()
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, *args, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.cpu().numpy(), orc.grouped_gemm_w4a4(ac, as_, aS, w[0], w[1], w[2], offs), "after timeout")
    assert sum(counts) == 8


def _drop_stage_zero(fn):
    os.environ["NVFP4MOE_TEST_DROP_STAGE"] = "0"
    try:
        t0 = time.time()
        fn()
        torch.cuda.synchronize()
        return time.time() - t0
    finally:
        del os.environ["NVFP4MOE_TEST_DROP_STAGE"]


def test_w4a16_gemm_bounded_wait_times_out_and_context_survives(orc):
    dev = cuda_or_skip()
    E, N, K = 2, 128, 512
    offs = np.array([0, 5, 8], np.int32)
    w = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w2", e, N, K).numpy() for e in range(E)]))
    a = wl.random_fp32((8, K), seed=2, tag="fail16").to(torch.bfloat16).float().numpy()
    wd = upload_weights(w, E, N, K, dev)
    args = (to_dev(a, dev, torch.bfloat16), None, None, *wd, to_dev(offs, dev), N, K)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    elapsed = _drop_stage_zero(lambda: B.moe_grouped_gemm_nvfp4(B.MOE_W4A16, *args, dev_status=status))
    assert int(status.item()) == NVFP4_E_DEVICE_TIMEOUT
    assert elapsed < 30.0
    status.zero_()
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A16, *args, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.cpu().numpy(), orc.grouped_gemm_w4a16(a, w[0], w[1], w[2], offs), "w4a16 after timeout")


def test_router_gemm_bounded_wait_times_out_and_context_survives(orc):
    dev = cuda_or_skip()
    T, H, E = 16, 1024, 256
    x = wl.activations_bf16(T, H, seed=4)
    wr = wl.router_weight_bf16(E, H, seed=4)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    elapsed = _drop_stage_zero(lambda: B.moe_router_logits(x.to(dev), wr.to(dev), dev_status=status))
    assert int(status.item()) == NVFP4_E_DEVICE_TIMEOUT
    assert elapsed < 30.0
    status.zero_()
    got = B.moe_router_logits(x.to(dev), wr.to(dev), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(got.cpu().numpy(), orc.router_logits(x.float().numpy(), wr.float().numpy()), "router after timeout")


@pytest.mark.parametrize("mode", ["w4a4", "w4a16"])
@pytest.mark.parametrize("drop", [0, 3])
def test_layer_bounded_wait_times_out_and_context_survives(orc, mode, drop):
    """The whole layer (its kernels chained as programmatic dependents): a GEMM
    stage that is never armed -- the first one, or one inside the first ring
    lap (H = 2048: four K stages per gate_up work unit after the split) --
    ends in a reported timeout, the kernels after it still run and return,
    and the next layer call gives the oracle's result."""
    dev = cuda_or_skip()
    cfg = wl.MoEConfig("fail_layer", T=8, H=2048, I=512, E=4, k=2, routing="uniform")
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
    os.environ["NVFP4MOE_TEST_DROP_STAGE"] = str(drop)
    try:
        t0 = time.time()
        B.moe_layer_forward(m, x, lg, cfg.k, g13, g2, S_h, dev_status=status)
        torch.cuda.synchronize()
        elapsed = time.time() - t0
    finally:
        del os.environ["NVFP4MOE_TEST_DROP_STAGE"]
    assert int(status.item()) == NVFP4_E_DEVICE_TIMEOUT
    assert elapsed < 30.0
    status.zero_()
    out = B.moe_layer_forward(m, x, lg, cfg.k, g13, g2, S_h, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = orc.moe_layer(mode, xt.float().numpy(), logits.numpy(), cfg.k, w13, w2, cfg.S_h)
    assert_close(out.cpu().numpy(), ref, "layer %s after timeout (drop %d)" % (mode, drop))
