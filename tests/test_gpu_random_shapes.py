"""Property tests: the grouped GEMM on seeded random shapes and routings.

Each case draws the expert count E, N (a multiple of 128), K (a multiple of
256) and per-expert row counts from a mix of empty experts, single rows,
partial and full 32-token groups and experts that take several 128-token
passes.  The draws land in both pass geometries (32- and 128-token passes)
and in the K-split launches (fewer work items than SMs).  The GEMM in NVFP4
W4A4, MXFP4 and W4A16 mode is compared with the oracle's fp64 grouped GEMM
on identical inputs, at the target's tolerances."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev, upload_weights
from test_gpu_mx import pad_scales, upload_mx_weights
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

N_CASES = 10


def _draw(case):
    """Case c % 3 == 0: sparse decode (0-4 rows per expert, at most one
    expert with up to 40); 1: a few dozen rows per expert; 2: a mix with
    experts of several 128-token passes."""
    rng = np.random.default_rng(7000 + case)
    E = int(rng.integers(2, 17))
    N = 128 * int(rng.integers(1, 5))
    K = 256 * int(rng.integers(1, 5))
    regime = case % 3
    if regime == 0:
        counts = rng.integers(0, 5, E)
        if rng.random() < 0.5:
            counts[int(rng.integers(0, E))] = int(rng.integers(5, 41))
    elif regime == 1:
        counts = rng.integers(0, 70, E)
    else:
        kind = rng.random(E)
        counts = np.where(kind < 0.2, 0,
                          np.where(kind < 0.5, rng.integers(1, 5, E),
                                   np.where(kind < 0.85, rng.integers(5, 70, E), rng.integers(129, 300, E))))
    if counts.sum() == 0:
        counts[int(rng.integers(0, E))] = int(rng.integers(1, 40))
    return counts.astype(np.int64), N, K


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def test_draws_cover_both_geometries_and_empty_experts():
    """The seeded draws include experts with no rows, passes of 32 tokens
    (R <= 4E) and of 128, and multi-pass experts (CPU-side check of the
    generator; runs with the GPU tests)."""
    draws = [_draw(c) for c in range(N_CASES)]
    assert any((c == 0).any() for c, _, _ in draws)
    assert any(c.sum() <= 4 * len(c) for c, _, _ in draws)
    assert any(c.sum() > 4 * len(c) for c, _, _ in draws)
    assert any(c.max() > 128 for c, _, _ in draws)


@pytest.mark.parametrize("case", range(N_CASES))
@pytest.mark.parametrize("mode", ["w4a4", "mxw4a4", "w4a16"])
def test_grouped_gemm_random_shape(orc, mode, case):
    dev = cuda_or_skip()
    counts, N, K = _draw(case)
    E = len(counts)
    offs = _offsets(counts)
    R = int(offs[-1])
    W = np.stack([wl.expert_weight_fp32("w13", e, N, K, 300 + case).numpy() for e in range(E)])
    a = wl.random_fp32((R, K), seed=400 + case, tag="acts").to(torch.bfloat16).float().numpy()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    if mode == "w4a4":
        w = orc.quantize_experts(W)
        ac, as_, aS = orc.quantize(a)
        ref = orc.grouped_gemm_w4a4(ac, as_, aS, w[0], w[1], w[2], offs)
        wd = upload_weights(w, E, N, K, dev)
        out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, to_dev(ac, dev), to_dev(as_, dev), to_dev(np.array([aS]), dev),
                                       wd[0], wd[1], wd[2], to_dev(offs, dev), N, K, dev_status=status)
    elif mode == "mxw4a4":
        w = orc.mx_quantize_experts(W)
        ac, as_ = orc.mx_quantize(a)
        ref = orc.grouped_gemm_mx(ac, as_, w[0], w[1], offs)
        wd = upload_mx_weights(w, E, N, K, dev)
        out = B.moe_grouped_gemm_nvfp4(B.MOE_MXW4A4, to_dev(ac, dev), to_dev(pad_scales(as_, K), dev), None, *wd,
                                       to_dev(offs, dev), N, K, dev_status=status)
    else:
        w = orc.quantize_experts(W)
        ref = orc.grouped_gemm_w4a16(a, w[0], w[1], w[2], offs)
        wd = upload_weights(w, E, N, K, dev)
        out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A16, to_dev(a, dev, torch.bfloat16), None, None, wd[0], wd[1], wd[2],
                                       to_dev(offs, dev), N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.cpu().numpy(), ref, "%s case %d (E=%d N=%d K=%d R=%d)" % (mode, case, E, N, K, R))
