"""GPU parity of the CTA-pair grouped GEMM (the .cta_group::2 kernel that
moe_grouped_gemm_nvfp4 runs when the experts see at least 1024 rows on
average and N % 256 == 0) against the oracle's fp64 grouped GEMM, NVFP4 and
MXFP4: one K stage, ragged last passes, an empty expert, K splits in two,
three and four parts and the unsplit many-tiles-per-pair schedule; and routing errors reported
through the status word."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev, upload_weights
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl
from test_gpu_mx import pad_scales, upload_mx_weights

pytestmark = pytest.mark.gpu

CASES = [
    # (counts per expert, N, K): all with >= 1024 rows per expert on average
    ([1024], 256, 256),              # four full passes, one K stage (no split)
    ([1100], 512, 1024),             # ragged last pass (1100 = 4 x 256 + 76), K in two parts
    ([1100, 0, 2000], 512, 1280),    # an empty expert; K in two parts of 2 and 3 stages
    ([2100, 2200], 4096, 512),       # 304 pair tiles, several per pair, no split
    ([2048], 512, 2048),             # 16 pair tiles: K in four parts of 2 stages
    ([1500, 700], 256, 1536),        # ragged passes of two experts: K in three parts
]


def _offsets(counts):
    return np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)


def _acts(R, K, seed):
    return wl.random_fp32((R, K), seed=seed, tag="pair").to(torch.bfloat16).float().numpy()


@pytest.mark.parametrize("case", range(len(CASES)))
def test_pair_gemm_nvfp4(orc, case):
    dev = cuda_or_skip()
    counts, N, K = CASES[case]
    E = len(counts)
    offs = _offsets(counts)
    R = int(offs[-1])
    w = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w13", e, N, K, 30 + case).numpy() for e in range(E)]))
    ac, as_, aS = orc.quantize(_acts(R, K, seed=300 + case))
    ref = orc.grouped_gemm_w4a4(ac, as_, aS, w[0], w[1], w[2], offs)
    wd = upload_weights(w, E, N, K, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, to_dev(ac, dev), to_dev(as_, dev), to_dev(np.array([aS]), dev),
                                   wd[0], wd[1], wd[2], to_dev(offs, dev), N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.cpu().numpy(), ref, "pair nvfp4 case %d" % case)


@pytest.mark.parametrize("case", [1, 3, 5])
def test_pair_gemm_mxfp4(orc, case):
    dev = cuda_or_skip()
    counts, N, K = CASES[case]
    E = len(counts)
    offs = _offsets(counts)
    R = int(offs[-1])
    w = orc.mx_quantize_experts(np.stack([wl.expert_weight_fp32("w2", e, N, K, 40 + case).numpy()
                                          for e in range(E)]))
    ac, as_ = orc.mx_quantize(_acts(R, K, seed=400 + case))
    ref = orc.grouped_gemm_mx(ac, as_, w[0], w[1], offs)
    wd = upload_mx_weights(w, E, N, K, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_MXW4A4, to_dev(ac, dev), to_dev(pad_scales(as_, K), dev), None, *wd,
                                   to_dev(offs, dev), N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.cpu().numpy(), ref, "pair mxfp4 case %d" % case)


def test_pair_gemm_bad_offsets_report_status():
    """Inconsistent offsets are reported through dev_status, not trapped."""
    dev = cuda_or_skip()
    E, N, K, R = 2, 256, 256, 2100
    wc = torch.zeros(E, N, K // 2, dtype=torch.uint8, device=dev)
    ws = torch.zeros(E * N * K // 16, dtype=torch.uint8, device=dev)
    wS = torch.ones(E, device=dev)
    a = torch.zeros(R, K // 2, dtype=torch.uint8, device=dev)
    asc = torch.zeros(R, K // 16, dtype=torch.uint8, device=dev)
    aS = torch.ones(1, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    offs = torch.tensor([0, 1400, 1300], dtype=torch.int32, device=dev)  # last != R, and decreasing
    B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, a, asc, aS, wc, ws, wS, offs, N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 8  # NVFP4_E_BAD_ROUTING
