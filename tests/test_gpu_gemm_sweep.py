"""Single-expert NVFP4 GEMM sweep (N=2048, K=6144, M in {1,16,64,512,4096}):
the shape of the pages' FP4 GEMM measurements ("The 2x Gap", sections "The
Investigation So Far" and "The Pivot": M=512, N=2048, K=6144; M=16-64 per
expert).  Activations N(0,1) and weights N(0,0.02) are quantised on the GPU
and by the oracle (bit-exact), then the GEMM runs through the grouped entry
point with one expert.  Rows are compared with the oracle in full up to
M=512, and at M=4096 on every row next to a 128-row tile boundary plus a
seeded spread (625 rows)."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

N, K = wl.GEMM_SWEEP["N"], wl.GEMM_SWEEP["K"]


@pytest.fixture(scope="module")
def weights(orc):
    dev = cuda_or_skip()
    _, w = wl.gemm_operands_fp32(1, N, K, device=dev)
    wc, ws, wS = B.nvfp4_quantize(w)
    oc, os_, oS = orc.quantize(w.cpu().numpy())
    torch.cuda.synchronize()
    assert np.array_equal(wc.cpu().numpy(), oc) and np.array_equal(ws.cpu().numpy(), os_)
    assert float(wS.item()) == float(oS)
    packed = B.nvfp4_pack_weight_scales(ws, 1, N, K)
    return (wc.view(1, N, K // 2), packed, wS), (oc[None], os_[None], np.array([oS], np.float32))


def _rows(M):
    """Every row up to M = 512; at larger M the two rows on each side of
    every 128-row boundary (tile edges of every geometry the kernels use)
    plus a seeded spread of 512 (625 rows at M = 4096)."""
    if M <= 512:
        return np.arange(M)
    edges = np.arange(0, M, 128)
    near = np.concatenate([edges - 2, edges - 1, edges, edges + 1])
    spread = np.random.default_rng(M).choice(M, 512, replace=False)
    r = np.unique(np.concatenate([near, spread, [M - 1]]))
    return r[(r >= 0) & (r < M)]


@pytest.mark.parametrize("M", wl.GEMM_SWEEP["Ms"])
def test_gemm_sweep(orc, weights, M):
    dev = cuda_or_skip()
    gw, ow = weights
    a, _ = wl.gemm_operands_fp32(M, 1, K, device=dev)
    ac, as_, aS = B.nvfp4_quantize(a)
    offs = torch.tensor([0, M], dtype=torch.int32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A4, ac, as_, aS, *gw, offs, N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = _rows(M)
    oac, oas, oaS = orc.quantize(a.cpu().numpy())
    assert np.array_equal(ac.cpu().numpy(), oac) and np.array_equal(as_.cpu().numpy(), oas)
    assert float(aS.item()) == float(oaS)
    ref = orc.grouped_gemm_w4a4(oac[rows], oas[rows], oaS, *ow, np.array([0, len(rows)], np.int32))
    assert_close(out.cpu().numpy()[rows], ref, "M=%d" % M)
