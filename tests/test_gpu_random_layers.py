"""Property tests: the whole layer on seeded random shapes against the oracle.

Each case draws T, H, I, E, k and the routing (uniform or Zipf) within the
library's constraints (H and I multiples of 256, k <= min(E, 8)).  The layer
runs through the staged entry points and through moe_layer_forward, which
must agree bit for bit; the staged intermediates and the output are then
compared with the oracle for every token, in W4A4, W4A16 and MXFP4, by the
same rules as the full-size layer tests (routing and the requantised codes
exactly, up to codes on a rounding boundary; outputs at the target's
tolerances)."""
import numpy as np
import pytest
import torch

from gpu_helpers import cuda_or_skip
from layer_parity import check_layer
from test_gpu_layer import MODES, gpu_weights, staged
from test_gpu_mx import gpu_mx_weights, staged_mx
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

N_CASES = 6


def _k_parts(R, E, N, K, sms):
    """K parts of the one-CTA grouped GEMM for this problem, as its launcher
    chooses them: passes of 32 tokens when R <= 4E (else 128), and K split
    while every part of every possible work item still fits in one wave."""
    tok = 32 if R <= 4 * E else 128
    items = (N // 128) * ((R + E * (tok - 1)) // tok)
    parts = 1
    while parts < 8 and items * (parts + 1) <= sms and K // 256 >= parts + 1:
        parts += 1
    return parts


def _assert_same_layer(fused, staged_out, cfg, mode, dev):
    """moe_layer_forward against the staged calls: bit for bit, except where
    a W4A4/MXFP4 GEMM adds more than two K parts, whose fp32 sums then follow
    the parts' arrival order; there the two may differ by summation rounding
    only (a wrong row would be off by the size of the output itself).  The
    dequantising W4A16 GEMM does not split K."""
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    parts = 1
    if mode != "w4a16":
        parts = max(_k_parts(cfg.R, cfg.E, 2 * cfg.I, cfg.H, sms), _k_parts(cfg.R, cfg.E, cfg.H, cfg.I, sms))
    if parts <= 2:
        assert torch.equal(fused, staged_out), "moe_layer_forward differs from the staged calls"
        return
    f, g = fused.double().cpu().numpy(), staged_out.double().cpu().numpy()
    rms = np.sqrt(np.mean(g ** 2))
    diff = np.abs(f - g).max() / rms
    print("\n%s: %d K parts, one-call vs staged max |diff| / RMS = %.2e" % (cfg.name, parts, diff))
    assert diff <= 1e-5, diff


def _cfg(case):
    rng = np.random.default_rng(9100 + case)
    E = int(rng.integers(2, 41))
    k = int(rng.integers(1, min(E, 8) + 1))
    T = int(rng.integers(1, 49))
    H = 256 * int(rng.integers(1, 5))
    I = 256 * int(rng.integers(1, 5))
    routing = "zipf" if rng.random() < 0.4 else "uniform"
    return wl.MoEConfig("random%d" % case, T=T, H=H, I=I, E=E, k=k, routing=routing)


@pytest.mark.parametrize("case", range(N_CASES))
@pytest.mark.parametrize("mode", ["w4a4", "w4a16", "mxw4a4"])
def test_layer_random_shape(orc, mode, case):
    dev = cuda_or_skip()
    cfg = _cfg(case)
    x = wl.activations_bf16(cfg.T, cfg.H, seed=case, device=dev)
    logits = wl.router_logits(cfg, seed=case, device=dev)
    if mode == "mxw4a4":
        (g13, l13), (g2, l2) = gpu_mx_weights(cfg, dev)
        d = staged_mx(x, logits, cfg, g13, g2)
        fused = B.moe_layer_forward(B.MOE_MXW4A4, x, logits, cfg.k, g13, g2, None)
        gw = ((g13[0], l13), (g2[0], l2))
    else:
        (g13, s13), (g2, s2) = gpu_weights(cfg, dev)
        S_h = torch.tensor([cfg.S_h], dtype=torch.float32, device=dev)
        d = staged(MODES[mode], x, logits, cfg, g13, g2, S_h)
        fused = B.moe_layer_forward(MODES[mode], x, logits, cfg.k, g13, g2, S_h)
        gw = ((g13[0], s13), (g2[0], s2))
    torch.cuda.synchronize()
    _assert_same_layer(fused, d["out"], cfg, mode, dev)
    check_layer(orc, cfg, mode, d, x, logits, gw, device=dev)
