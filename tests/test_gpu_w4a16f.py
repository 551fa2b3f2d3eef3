"""GPU checks of the F16 carrier of W4A16 (moe_gather_f16, moe_swiglu_f16)
and of the grouped GEMM on it (MOE_W4A16F).

The carrier holds each bf16 row as f16(x * 2^e_r) with 2^-e_r beside it.
What the header promises is checked element by element: 2^-e_r is a power
of two placing the row's max in [2^14, 2^15) (1 for a zero row); every
element that lands on an f16 normal comes back exactly (f16 * 2^-e_r == x);
the others are within half an f16 subnormal step.  The GEMM on the carrier
is compared with the oracle's fp64 W4A16 GEMM on the bf16 values, and with
the BF16 form of the same kernel."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev, upload_weights
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

F16_MIN_NORMAL = 2.0 ** -14


def _rows_with_extremes(T, H, seed):
    """bf16 rows of very different magnitudes: N(0,1), huge, tiny, one of
    zeros, and rows whose values span 60 binary orders of magnitude."""
    x = wl.random_fp32((T, H), seed=seed, tag="f16carrier")
    g = torch.Generator().manual_seed(seed)
    x[1] *= 1e30
    x[2] *= 1e-30
    x[3] = 0.0
    span = torch.pow(2.0, torch.randint(-40, 20, (H,), generator=g).float())
    x[4] *= span
    x[5] = x[4] * 3.0e12
    return x.to(torch.bfloat16)


def _check_carrier(src_bf16, a_f16, rs):
    """src_bf16 [R, H] (the bf16 rows carried), a_f16 [R, H], rs [R]."""
    x = src_bf16.float().cpu().numpy().astype(np.float64)
    a = a_f16.float().cpu().numpy().astype(np.float64)
    s = rs.cpu().numpy().astype(np.float64)
    m, e = np.frexp(s)
    assert (m == 0.5).all(), "row multipliers are not powers of two"
    amax = np.abs(x).max(axis=1)
    for r in range(x.shape[0]):
        if amax[r] == 0:
            assert s[r] == 1.0 and (a[r] == 0).all()
            continue
        scaled_max = amax[r] / s[r]
        # the largest magnitude lands in [2^14, 2^15) unless the exponent was capped
        assert scaled_max < 2.0 ** 15, (r, scaled_max)
        assert scaled_max >= 2.0 ** 14 or s[r] == 2.0 ** -126, (r, scaled_max)
    back = a * s[:, None]
    normal = np.abs(a) >= F16_MIN_NORMAL
    assert np.array_equal(back[normal], x[normal]), "an f16-normal element did not come back exactly"
    err = np.abs(back - x)[~normal]
    bound = (2.0 ** -25 * np.broadcast_to(s[:, None], x.shape))[~normal]
    assert (err <= bound).all(), "a subnormal-range element is off by more than half an f16 step"


def test_gather_f16_rows_exact():
    dev = cuda_or_skip()
    T, H = 40, 512
    x = _rows_with_extremes(T, H, seed=11).to(dev)
    g = torch.Generator().manual_seed(3)
    perm = torch.randint(0, T, (3 * T,), generator=g, dtype=torch.int32)
    perm[:T] = torch.arange(T, dtype=torch.int32)  # every row at least once
    a, rs = B.moe_gather_f16(x, perm.to(dev))
    torch.cuda.synchronize()
    _check_carrier(x[perm.to(dev).long()], a, rs)
    # without a permutation: rows in order
    a2, rs2 = B.moe_gather_f16(x)
    torch.cuda.synchronize()
    _check_carrier(x, a2, rs2)


def test_swiglu_f16_carries_the_bf16_swiglu():
    dev = cuda_or_skip()
    R, I = 70, 512
    G = wl.random_fp32((R, 2 * I), seed=5, tag="swiglu_f16").to(dev) * 4.0
    G[3] *= 1e-20  # a row of tiny h
    G[4, :I] = -200.0  # silu saturates to -0.0: h is a row of signed zeros
    hb = B.moe_swiglu_requant(G, B.MOE_W4A16)
    hf, rs = B.moe_swiglu_f16(G)
    torch.cuda.synchronize()
    _check_carrier(hb, hf, rs)


CASES = [([3, 0, 17, 1, 40], 256, 512), ([1] * 16, 512, 1024), ([70, 2], 384, 2048)]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_gemm_w4a16f_against_oracle_and_bf16_form(orc, case):
    dev = cuda_or_skip()
    counts, N, K = CASES[case]
    E = len(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offs[-1])
    w = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w13", e, N, K, 40 + case).numpy() for e in range(E)]))
    xb = wl.random_fp32((R, K), seed=400 + case, tag="w4a16f").to(torch.bfloat16)
    xb[0] *= 1e3
    ref = orc.grouped_gemm_w4a16(xb.float().numpy(), w[0], w[1], w[2], offs)
    wd = upload_weights(w, E, N, K, dev)
    xd = xb.to(dev)
    a, rs = B.moe_gather_f16(xd)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    got = B.moe_grouped_gemm_nvfp4(B.MOE_W4A16F, a, None, rs, wd[0], wd[1], wd[2], to_dev(offs, dev), N, K,
                                   dev_status=status)
    bf = B.moe_grouped_gemm_nvfp4(B.MOE_W4A16, xd, None, None, wd[0], wd[1], wd[2], to_dev(offs, dev), N, K)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(got.cpu().numpy(), ref, "w4a16f case %d" % case)
    # the same products, summed in the same order by the same kernel: the
    # two forms agree to the last bits
    g64, b64 = got.double().cpu().numpy(), bf.double().cpu().numpy()
    scale = np.abs(b64).max()
    assert np.abs(g64 - b64).max() <= 1e-6 * scale, np.abs(g64 - b64).max() / scale
