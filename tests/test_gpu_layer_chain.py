"""Back-to-back layers whose routing changes from call to call.

Inside moe_layer_forward the W4A4 and MXFP4 grouped GEMMs read the routing
(expert_offsets) and start their weight copies before their grid-dependency
wait, relying on the routing having been written by an earlier kernel of the
same call.  Here several layer calls with alternating router logits share one
workspace and are enqueued without any synchronisation in between (directly
on a stream, and as one replayed CUDA graph), so a GEMM that read the
previous call's routing would compute wrong rows.  Every output must equal,
bit for bit, the same call run alone.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import cuda_or_skip
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

# (T, H, I, E, k): 32-token passes (R <= 4E), and 128-token passes with
# experts holding ~60 rows
SHAPES = [(16, 1024, 512, 64, 8), (256, 1024, 512, 16, 4)]


def _weights(mode, cfg, dev):
    out = []
    for which, N, K in (("w13", 2 * cfg.I, cfg.H), ("w2", cfg.H, cfg.I)):
        codes = torch.empty(cfg.E, N, K // 2, dtype=torch.uint8, device=dev)
        if mode == B.MOE_MXW4A4:
            lin = torch.empty(cfg.E, N, K // 32, dtype=torch.uint8, device=dev)
            for e in range(cfg.E):
                _, s = B.mxfp4_quantize(wl.expert_weight_fp32(which, e, N, K, 3, device=dev), codes=codes[e])
                lin[e].copy_(s[:, : K // 32])
            out.append((codes, B.mxfp4_pack_weight_scales(lin, cfg.E, N, K), None))
        else:
            scales = torch.empty(cfg.E, N, K // 16, dtype=torch.uint8, device=dev)
            S = torch.empty(cfg.E, dtype=torch.float32, device=dev)
            for e in range(cfg.E):
                _, _, s = B.nvfp4_quantize(wl.expert_weight_fp32(which, e, N, K, 3, device=dev), codes=codes[e],
                                           scales=scales[e])
                S[e:e + 1].copy_(s)
            out.append((codes, B.nvfp4_pack_weight_scales(scales, cfg.E, N, K), S))
    return out


@pytest.mark.parametrize("mode", [B.MOE_W4A4, B.MOE_MXW4A4], ids=["w4a4", "mxw4a4"])
@pytest.mark.parametrize("shape", range(len(SHAPES)))
def test_alternating_routings_share_a_workspace(mode, shape):
    dev = cuda_or_skip()
    T, H, I, E, k = SHAPES[shape]
    cfg = wl.MoEConfig("chain", T=T, H=H, I=I, E=E, k=k, routing="uniform")
    w13, w2 = _weights(mode, cfg, dev)
    S_h = torch.tensor([cfg.S_h], dtype=torch.float32, device=dev)
    x = wl.activations_bf16(T, H, seed=5, device=dev)
    logits = [wl.router_logits(cfg, seed=s, device=dev) for s in (11, 12)]
    ws = torch.empty(B.moe_layer_workspace_bytes(mode, T, H, I, E, k), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)

    # each routing alone, with a synchronisation after the call
    alone = []
    for lg in logits:
        alone.append(B.moe_layer_forward(mode, x, lg, k, w13, w2, S_h, workspace=ws, dev_status=status).clone())
        torch.cuda.synchronize()
    assert int(status.item()) == 0
    ids = [torch.topk(lg, k, dim=1).indices.sort(dim=1).values for lg in logits]
    assert not torch.equal(ids[0], ids[1]), "the two routings should differ"

    # back to back on the stream, one shared workspace
    n = 6
    outs = [torch.empty(T, H, dtype=torch.float32, device=dev) for _ in range(n)]
    for i in range(n):
        B.moe_layer_forward(mode, x, logits[i % 2], k, w13, w2, S_h, out=outs[i], workspace=ws, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for i in range(n):
        assert torch.equal(outs[i], alone[i % 2]), "call %d differs from the same routing run alone" % i

    # the same chain captured once and replayed twice
    for o in outs:
        o.zero_()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            B.moe_layer_forward(mode, x, logits[i % 2], k, w13, w2, S_h, out=outs[i], workspace=ws,
                                dev_status=status)
    for _ in range(2):
        g.replay()
        torch.cuda.synchronize()
        for i in range(n):
            assert torch.equal(outs[i], alone[i % 2]), "graph replay: call %d differs" % i
    assert int(status.item()) == 0
    assert np.isfinite(alone[0].cpu().numpy()).all()
