"""More work units per CTA than the grouped GEMMs' prologue tables hold (256
per CTA; the ones beyond are decoded on the fly inside the main loop).

One expert, N = 128, K = 256 and SMs x 257 x 128 token rows give one unit per
128-token pass, so every CTA runs at least 257 units.  Activations are random
codes and scales generated on the GPU (any byte is a valid E2M1 pair).  Rows
from the first units, from units 255-257 of the first and last CTA, and the
last rows are checked against fp64 dot products of the operands decoded with
the oracle's format tables."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev, upload_weights
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

N, K = 128, 256


def _setup(orc, dev):
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    R = sms * 257 * 128
    W = wl.expert_weight_fp32("w13", 0, N, K, 21).numpy()[None]
    w = orc.quantize_experts(W)
    wd = upload_weights(w, 1, N, K, dev)
    wdeq = orc.dequantize(w[0][0], w[1][0], 1.0, K) * np.float64(w[2][0])
    offs = torch.tensor([0, R], dtype=torch.int32, device=dev)
    rows = sorted({0, 1, 127, 128, R - 1, R - 128})
    for c in (0, sms - 1):
        for j in (255, 256, 257):
            u = c + j * sms
            rows += [u * 128, u * 128 + 77, u * 128 + 127]
    return sms, R, wd, wdeq, offs, sorted(set(r for r in rows if r < R))


def test_gemm_w4a4_more_units_than_the_table(orc):
    dev = cuda_or_skip()
    sms, R, wd, wdeq, offs, rows = _setup(orc, dev)
    g = torch.Generator(device=dev).manual_seed(5)
    codes = torch.randint(0, 256, (R, K // 2), dtype=torch.uint8, device=dev, generator=g)
    scales = torch.randint(0x28, 0x41, (R, K // 16), dtype=torch.uint8, device=dev, generator=g)
    aS = torch.ones(1, dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, codes, scales, aS, *wd, offs, N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    idx = torch.tensor(rows, device=dev)
    c = codes[idx].cpu().numpy()
    s = scales[idx].cpu().numpy()
    e2m1 = np.array([orc.e2m1_value(v) for v in range(16)])
    e4m3 = np.array([orc.e4m3_value(v) for v in range(256)])
    nib = np.stack([c & 15, c >> 4], -1).reshape(len(rows), K)
    a = e2m1[nib] * np.repeat(e4m3[s], 16, axis=1)
    ref = a @ wdeq.T
    got = out[idx].cpu().numpy()
    del out, codes, scales
    assert_close(got, ref, "w4a4, %d units per CTA" % (R // 128 // sms))


def test_gemm_w4a16_more_units_than_the_table(orc):
    dev = cuda_or_skip()
    sms, R, wd, wdeq, offs, rows = _setup(orc, dev)
    g = torch.Generator(device=dev).manual_seed(6)
    a = torch.randn(R, K, dtype=torch.float32, device=dev, generator=g).to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A16, a, None, None, *wd, offs, N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    idx = torch.tensor(rows, device=dev)
    ref = a[idx].double().cpu().numpy() @ wdeq.T
    got = out[idx].cpu().numpy()
    del out, a
    assert_close(got, ref, "w4a16, %d units per CTA" % (R // 128 // sms))
