"""Full MoE layer on the GPU against the oracle.

* tiny workload: every intermediate and the output, all tokens.
* decode workloads at full size, in the launch configuration the benchmark
  times (moe_layer_forward, checked bitwise against the staged entry points):
  EVERY token of the batch against the oracle -- decode_c16 (16 tokens),
  wide (64 tokens, 22 experts each) and decode_b512 (512 tokens, which covers
  every token routed to the heaviest Zipf experts) -- with the same fp32
  weights (regenerated from their seeds, quantised by the oracle and checked
  bit-exact against the GPU's quantisation) and the whole batch's activation
  scale.  The tolerances, the treatment of requantised h codes that sit on a
  rounding boundary, and the figures printed are described in layer_parity.
"""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, nvfp4_ambiguous, unpack_codes, upload_weights
from layer_parity import FLIP_WINDOW, check_layer
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _oracle_weights(orc, cfg, experts, seed=0, device="cpu"):
    """fp32 weights from their seeds (on `device`, the generator the GPU side
    used), quantised by the oracle."""
    w13 = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w13", e, 2 * cfg.I, cfg.H, seed, device).cpu().numpy()
                                         for e in experts]))
    w2 = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w2", e, cfg.H, cfg.I, seed, device).cpu().numpy()
                                        for e in experts]))
    return w13, w2


def gpu_weights(cfg, dev, seed=0):
    """Quantise every expert on the GPU (product quantiser), pack scales."""
    out = []
    for which, N, K in (("w13", 2 * cfg.I, cfg.H), ("w2", cfg.H, cfg.I)):
        codes = torch.empty(cfg.E, N, K // 2, dtype=torch.uint8, device=dev)
        scales = torch.empty(cfg.E, N, K // 16, dtype=torch.uint8, device=dev)
        S = torch.empty(cfg.E, dtype=torch.float32, device=dev)
        for e in range(cfg.E):
            wf = wl.expert_weight_fp32(which, e, N, K, seed, device=dev)
            _, _, s = B.nvfp4_quantize(wf, codes=codes[e], scales=scales[e])
            S[e:e + 1].copy_(s)
        packed = B.nvfp4_pack_weight_scales(scales, cfg.E, N, K)
        out.append(((codes, packed, S), scales))
    return out


def staged(mode, x, logits, cfg, w13, w2, S_h):
    """The layer through the individual entry points (exposes intermediates)."""
    k, I, H = cfg.k, cfg.I, cfg.H
    R = cfg.R
    d = {}
    if mode == B.MOE_W4A4:
        xc, xs, S_x = B.nvfp4_quantize(x)
        rt = B.moe_align_permute(logits, k, act=(xc, xs), act_kind=B.MOE_ACT_NVFP4)
        G = B.moe_grouped_gemm_nvfp4(mode, rt["act_codes"], rt["act_scales"], S_x, *w13, rt["offsets"], 2 * I, H)
        hc, hs = B.moe_swiglu_requant(G, mode, S_h)
        Y = B.moe_grouped_gemm_nvfp4(mode, hc, hs, S_h, *w2, rt["offsets"], H, I)
        d.update(S_x=S_x, hc=hc, hs=hs)
    else:
        # W4A16 as moe_layer_forward runs it: the bf16 operands carried as F16
        # rows (moe_gather_f16, moe_swiglu_f16) into the MOE_W4A16F GEMMs
        rt = B.moe_align_permute(logits, k)
        a, a_rs = B.moe_gather_f16(x, rt["perm"])
        G = B.moe_grouped_gemm_nvfp4(B.MOE_W4A16F, a, None, a_rs, *w13, rt["offsets"], 2 * I, H)
        hf, h_rs = B.moe_swiglu_f16(G)
        Y = B.moe_grouped_gemm_nvfp4(B.MOE_W4A16F, hf, None, h_rs, *w2, rt["offsets"], H, I)
        d.update(hb=(hf.float() * h_rs[:, None]).to(torch.bfloat16))
    out = B.moe_combine(Y, rt["inv"], rt["w"])
    d.update(rt=rt, G=G, Y=Y, out=out)
    return d


MODES = {"w4a4": B.MOE_W4A4, "w4a16": B.MOE_W4A16}


@pytest.mark.parametrize("mode", ["w4a4", "w4a16"])
def test_layer_tiny_all_intermediates(orc, mode):
    dev = cuda_or_skip()
    cfg = wl.CONFIGS["tiny"]
    m = MODES[mode]
    xt = wl.activations_bf16(cfg.T, cfg.H)
    logits = wl.router_logits(cfg)
    w13, w2 = _oracle_weights(orc, cfg, range(cfg.E))
    ref, mids = orc.moe_layer(mode, xt.float().numpy(), logits.numpy(), cfg.k, w13, w2, cfg.S_h, intermediates=True)
    g13 = upload_weights(w13, cfg.E, 2 * cfg.I, cfg.H, dev)
    g2 = upload_weights(w2, cfg.E, cfg.H, cfg.I, dev)
    S_h = torch.tensor([cfg.S_h], dtype=torch.float32, device=dev)
    x, lg = xt.to(dev), logits.to(dev)
    d = staged(m, x, lg, cfg, g13, g2, S_h)
    fused = B.moe_layer_forward(m, x, lg, cfg.k, g13, g2, S_h)
    torch.cuda.synchronize()
    assert torch.equal(fused, d["out"])
    assert np.array_equal(d["rt"]["ids"].cpu().numpy(), mids["ids"])
    assert np.array_equal(d["rt"]["offsets"].cpu().numpy(), mids["offsets"])
    assert np.array_equal(d["rt"]["perm"].cpu().numpy(), mids["perm"])
    assert np.array_equal(d["rt"]["inv"].cpu().numpy(), mids["inv"])
    if mode == "w4a4":
        assert float(d["S_x"].item()) == float(mids["S_x"])
        amb = nvfp4_ambiguous(mids["h32"], cfg.S_h, rel=FLIP_WINDOW)
        flips = unpack_codes(d["hc"].cpu().numpy()) != unpack_codes(mids["hq_codes"])
        assert not (flips & ~amb).any()
    assert_close(d["out"].cpu().numpy(), ref, "tiny " + mode)


def _full_check(orc, cfg, mode, dev, tokens=None):
    m = MODES[mode]
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    logits = wl.router_logits(cfg, device=dev)
    (g13, s13), (g2, s2) = gpu_weights(cfg, dev)
    S_h = torch.tensor([cfg.S_h], dtype=torch.float32, device=dev)
    d = staged(m, x, logits, cfg, g13, g2, S_h)
    fused = B.moe_layer_forward(m, x, logits, cfg.k, g13, g2, S_h)
    torch.cuda.synchronize()
    assert torch.equal(fused, d["out"]), "moe_layer_forward differs from the staged calls"
    return check_layer(orc, cfg, mode, d, x, logits, ((g13[0], s13), (g2[0], s2)), tokens=tokens, device=dev)


@pytest.mark.parametrize("mode", ["w4a4", "w4a16"])
def test_layer_decode_c16_full_size(orc, mode):
    dev = cuda_or_skip()
    _full_check(orc, wl.CONFIGS["decode_c16"], mode, dev)


@pytest.mark.parametrize("mode", ["w4a4", "w4a16"])
def test_layer_wide_full_size(orc, mode):
    dev = cuda_or_skip()
    _full_check(orc, wl.CONFIGS["wide"], mode, dev)


def test_layer_decode_b512_full_size(orc):
    dev = cuda_or_skip()
    _full_check(orc, wl.CONFIGS["decode_b512"], "w4a4", dev)


@pytest.mark.parametrize("mode", ["w4a4", "w4a16"])
def test_layer_graph_matches_one_call(orc, mode):
    """MoELayerGraph (moe_layer_forward_host from pinned host buffers,
    replayed as one CUDA graph) gives exactly moe_layer_forward's output, on
    two different inputs in a row."""
    dev = cuda_or_skip()
    cfg = wl.CONFIGS["decode_c16"]
    m = MODES[mode]
    (g13, _), (g2, _) = gpu_weights(cfg, dev)
    S_h = torch.tensor([cfg.S_h], dtype=torch.float32, device=dev)
    graph = B.MoELayerGraph(m, cfg.T, cfg.H, cfg.E, cfg.k, g13, g2, S_h, device=dev)
    for seed in (0, 1):
        x = wl.activations_bf16(cfg.T, cfg.H, seed=seed, device=dev)
        logits = wl.router_logits(cfg, seed=seed, device=dev)
        ref = B.moe_layer_forward(m, x, logits, cfg.k, g13, g2, S_h)
        torch.cuda.synchronize()
        got = graph.run(x.cpu(), logits.cpu())
        assert torch.equal(got, ref.cpu()), seed
        assert int(graph.dev_status.item()) == 0


@pytest.mark.parametrize("mode", ["w4a4", "w4a16", "mxw4a4", "w4a8"])
@pytest.mark.parametrize("shape", [(16, 4096, 2048, 256, 8), (3, 256, 512, 7, 2), (40, 1024, 256, 64, 4)])
def test_layer_host_entry_matches_device_entry(orc, mode, shape):
    """moe_layer_forward_host (inputs staged from pinned host memory by a
    kernel, output written to pinned host memory by the combine kernel) is
    bitwise moe_layer_forward on device copies of the same inputs -- also
    for a logits row of 7 experts (28 bytes: not a multiple of 16) and for
    more than one routing chunk (40 tokens)."""
    dev = cuda_or_skip()
    T, H, I, E, k = shape
    cfg = wl.MoEConfig("host_entry", T=T, H=H, I=I, E=E, k=k, routing="uniform")
    m = {"w4a4": B.MOE_W4A4, "w4a16": B.MOE_W4A16, "mxw4a4": B.MOE_MXW4A4, "w4a8": B.MOE_W4A8}[mode]
    if mode == "mxw4a4":
        from test_gpu_mx import gpu_mx_weights
        (g13, _), (g2, _) = gpu_mx_weights(cfg, dev)
    else:
        (g13, _), (g2, _) = gpu_weights(cfg, dev)
    S_h = torch.tensor([cfg.S_h], dtype=torch.float32, device=dev)
    x = wl.activations_bf16(T, H, seed=3, device=dev)
    logits = wl.router_logits(cfg, seed=3, device=dev)
    ref = B.moe_layer_forward(m, x, logits, k, g13, g2, S_h)
    xh = x.cpu().pin_memory()
    lh = logits.cpu().pin_memory()
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    got = B.moe_layer_forward_host(m, xh, lh, k, g13, g2, S_h, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(got, ref.cpu())



@pytest.mark.parametrize("mode", ["w4a4", "w4a16"])
@pytest.mark.parametrize("shape", [(5, 256, 256, 4, 4), (33, 256, 256, 1024, 32)])
def test_layer_degenerate_routing_against_oracle(orc, mode, shape):
    """Routing extremes through the whole layer: every token to every expert
    (k = E: the softmax covers all experts), and the largest expert count and
    top-k the entry points accept (E = 1024, k = 32) over two routing chunks
    (33 tokens), with most experts receiving one or two rows."""
    dev = cuda_or_skip()
    T, H, I, E, k = shape
    cfg = wl.MoEConfig("degenerate", T=T, H=H, I=I, E=E, k=k, routing="uniform")
    m = MODES[mode]
    xt = wl.activations_bf16(T, H, seed=7)
    logits = wl.router_logits(cfg, seed=7)
    w13, w2 = _oracle_weights(orc, cfg, range(E), seed=7)
    g13 = upload_weights(w13, E, 2 * I, H, dev)
    g2 = upload_weights(w2, E, H, I, dev)
    S_h = torch.tensor([cfg.S_h], dtype=torch.float32, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    got = B.moe_layer_forward(m, xt.to(dev), logits.to(dev), k, g13, g2, S_h, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = orc.moe_layer(mode, xt.float().numpy(), logits.numpy(), k, w13, w2, cfg.S_h)
    assert_close(got.cpu().numpy(), ref, "%s %s" % (mode, shape))


def test_layer_zero_tokens():
    """T = 0: nothing to do, no error, an empty output."""
    dev = cuda_or_skip()
    cfg = wl.CONFIGS["tiny"]
    (g13, _), (g2, _) = gpu_weights(cfg, dev)
    S_h = torch.tensor([cfg.S_h], dtype=torch.float32, device=dev)
    x = torch.empty(0, cfg.H, dtype=torch.bfloat16, device=dev)
    lg = torch.empty(0, cfg.E, dtype=torch.float32, device=dev)
    for m in (B.MOE_W4A4, B.MOE_W4A16):
        out = B.moe_layer_forward(m, x, lg, cfg.k, g13, g2, S_h)
        torch.cuda.synchronize()
        assert tuple(out.shape) == (0, cfg.H)
