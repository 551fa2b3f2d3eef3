"""GPU parity of moe_grouped_gemm_nvfp4 (W4A4 and W4A16) against the oracle's
fp64 grouped GEMM, on identical NVFP4 inputs, with ragged per-expert row
counts (empty experts, 1 row, partial 32-row groups, more than one 128-row
pass) and several K-chunks."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev, upload_weights
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _weights(orc, E, N, K, seed):
    w = np.stack([wl.expert_weight_fp32("w13", e, N, K, seed).numpy() for e in range(E)])
    return orc.quantize_experts(w)


def _acts(orc, R, K, seed):
    a = wl.random_fp32((R, K), seed=seed, tag="acts").to(torch.bfloat16).float().numpy()
    return a


CASES = [
    # (counts per expert, N, K)
    ([1], 128, 256),
    ([3, 0, 1, 7, 2], 256, 512),
    ([0, 31, 32, 33, 64, 1, 0, 65], 384, 256),
    ([129, 0, 200, 5], 128, 1024),
    ([16] * 12, 512, 768),
    # few tokens per expert on average (the 32-token-pass, 8-stage geometry),
    # with a 40-token expert taking two passes, and a K-split case
    ([40, 0, 0, 0, 0, 0, 0, 0, 0, 0, 1], 256, 512),
    ([2, 0, 3], 128, 1024),
]


@pytest.mark.parametrize("case", range(len(CASES)))
def test_gemm_w4a4_ragged(orc, case):
    dev = cuda_or_skip()
    counts, N, K = CASES[case]
    E = len(counts)
    offs = _offsets(counts)
    R = int(offs[-1])
    w = _weights(orc, E, N, K, seed=case)
    a = _acts(orc, R, K, seed=100 + case)
    ac, as_, aS = orc.quantize(a)
    ref = orc.grouped_gemm_w4a4(ac, as_, aS, w[0], w[1], w[2], offs)
    wd = upload_weights(w, E, N, K, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, to_dev(ac, dev), to_dev(as_, dev), to_dev(np.array([aS]), dev),
                                   wd[0], wd[1], wd[2], to_dev(offs, dev), N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.cpu().numpy(), ref, "w4a4 case %d" % case)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_gemm_w4a16_ragged(orc, case):
    dev = cuda_or_skip()
    counts, N, K = CASES[case]
    E = len(counts)
    offs = _offsets(counts)
    R = int(offs[-1])
    w = _weights(orc, E, N, K, seed=case)
    a = _acts(orc, R, K, seed=200 + case)
    ref = orc.grouped_gemm_w4a16(a, w[0], w[1], w[2], offs)
    wd = upload_weights(w, E, N, K, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A16, to_dev(a, dev, torch.bfloat16), None, None, wd[0], wd[1], wd[2],
                                   to_dev(offs, dev), N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.cpu().numpy(), ref, "w4a16 case %d" % case)


def test_gemm_w4a4_one_hot_exact(orc):
    """Rows with a single 1.0 pick out a weight column: exact, any order."""
    dev = cuda_or_skip()
    E, N, K = 2, 128, 512
    w = _weights(orc, E, N, K, seed=9)
    cols = [0, 1, 255, 256, 300, 511]
    R = len(cols)
    ac = np.zeros((R, K // 2), np.uint8)
    as_ = np.full((R, K // 16), 0x38, np.uint8)
    for r, c in enumerate(cols):
        ac[r, c // 2] = 2 << (4 * (c % 2))
    offs = _offsets([3, 3])
    ref = orc.grouped_gemm_w4a4(ac, as_, 1.0, w[0], w[1], w[2], offs)
    wd = upload_weights(w, E, N, K, dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, to_dev(ac, dev), to_dev(as_, dev), to_dev(np.ones(1, np.float32), dev),
                                   wd[0], wd[1], wd[2], to_dev(offs, dev), N, K)
    assert np.array_equal(out.cpu().numpy(), ref.astype(np.float32))


def test_gemm_bad_offsets_report_status():
    """Inconsistent offsets are reported through dev_status, not trapped."""
    dev = cuda_or_skip()
    E, N, K, R = 2, 128, 256, 8
    wc = torch.zeros(E, N, K // 2, dtype=torch.uint8, device=dev)
    ws = torch.zeros(E * N * K // 16, dtype=torch.uint8, device=dev)
    wS = torch.ones(E, device=dev)
    a = torch.zeros(R, K // 2, dtype=torch.uint8, device=dev)
    asc = torch.zeros(R, K // 16, dtype=torch.uint8, device=dev)
    aS = torch.ones(1, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    offs = torch.tensor([0, 5, 3], dtype=torch.int32, device=dev)  # last != R, and decreasing
    B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, a, asc, aS, wc, ws, wS, offs, N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 8  # NVFP4_E_BAD_ROUTING
