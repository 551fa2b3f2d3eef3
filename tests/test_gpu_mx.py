"""GPU parity of the MXFP4 path (group-32 blocks, UE8M0 scales) against the
oracle: the quantiser bit for bit, the grouped GEMM (kind::mxf4nvf4
.scale_vec::2X) on ragged expert groups, SwiGLU + requantisation, the fused
route + quantise front half, and the whole layer (tiny with every
intermediate; decode shapes at full size: every token of decode_c16 and wide, every
fourth token of decode_b512).

Where a requantised code of h differs, the oracle's own fp32 h must lie
within FLIP_WINDOW (relative, see layer_parity) of that code's rounding
midpoint or its block's amax that close to a power of two (the
shared-exponent boundary): G is accumulated in fp32 on the GPU and in fp64
in the oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev, unpack_codes
from layer_parity import FLIP_WINDOW, check_layer
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def pad_scales(s, cols):
    """Linear MXFP4 scales [rows, cols/32] -> the library's padded rows."""
    pitch = B.mxfp4_scale_pitch(cols)
    out = np.zeros((s.shape[0], pitch), np.uint8)
    out[:, : cols // 32] = s
    return out


def mx_ambiguous(v, rel=1e-5):
    """True where an element's E2M1 decision, or its block's shared exponent,
    lies within `rel` of a rounding boundary."""
    v = np.asarray(v, np.float64)
    rows, cols = v.shape
    amax = np.abs(v).reshape(rows, cols // 32, 32).max(-1)
    with np.errstate(divide="ignore"):
        lg = np.log2(np.where(amax > 0, amax, 1.0))
    near_pow2 = np.abs(amax - np.exp2(np.round(lg))) <= rel * np.maximum(amax, 1e-300)
    E = np.clip(np.floor(lg) - 2, -127, 127)
    q = np.abs(v) / np.repeat(np.exp2(E), 32, axis=1)
    e2 = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    near_el = np.min(np.abs(q[..., None] - e2), axis=-1) <= rel * np.maximum(q, 1e-30)
    return near_el | np.repeat(near_pow2, 32, axis=1)


def upload_mx_weights(w, E, N, K, device):
    """(codes, linear scales [E, N, K/32], None) numpy -> GPU (codes, packed, None)."""
    codes = to_dev(w[0], device)
    packed = B.mxfp4_pack_weight_scales(to_dev(w[1], device), E, N, K)
    return codes, packed, None


# ---------------------------------------------------------------------------
# quantiser
# ---------------------------------------------------------------------------

def _hard_inputs(rows, cols, seed):
    """Normal values over a wide exponent range, plus zero blocks, subnormals,
    exact E2M1 midpoints and exact powers of two."""
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-30, 30, (rows, 1)))
    x = x.astype(np.float32)
    if cols >= 64:
        x[0, 0:32] = 0.0
        x[0, 32:64] = np.float32(2.0 ** -140) * np.arange(32)  # subnormals, E clamps to -127
    if rows > 1:
        # amax 4 -> E = 0; elements on every E2M1 midpoint, both signs
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 4.0], np.float32)
        x[1, :16] = np.concatenate([mids, -mids])
        x[1, 16:32] = 0.5
    return x


@pytest.mark.parametrize("rows,cols", [(1, 32), (3, 96), (37, 512), (128, 4096), (5, 6144)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_mx_quantize_bit_exact(orc, rows, cols, dtype):
    dev = cuda_or_skip()
    x = torch.from_numpy(_hard_inputs(rows, cols, rows * cols)).to(dtype)
    codes, scales = B.mxfp4_quantize(x.to(dev))
    torch.cuda.synchronize()
    oc, os_ = orc.mx_quantize(x.float().numpy())
    assert np.array_equal(codes.cpu().numpy(), oc)
    s = scales.cpu().numpy()
    assert np.array_equal(s[:, : cols // 32], os_)
    assert not s[:, cols // 32:].any()  # padding is zero


# ---------------------------------------------------------------------------
# grouped GEMM
# ---------------------------------------------------------------------------

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
def test_mx_gemm_ragged(orc, case):
    dev = cuda_or_skip()
    counts, N, K = CASES[case]
    E = len(counts)
    offs = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    R = int(offs[-1])
    W = np.stack([wl.expert_weight_fp32("w13", e, N, K, 11 + case).numpy() for e in range(E)])
    w = orc.mx_quantize_experts(W)
    a = wl.random_fp32((R, K), seed=case, tag="acts").to(torch.bfloat16).float().numpy()
    ac, as_ = orc.mx_quantize(a)
    ref = orc.grouped_gemm_mx(ac, as_, w[0], w[1], offs)
    wd = upload_mx_weights(w, E, N, K, dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_MXW4A4, to_dev(ac, dev), to_dev(pad_scales(as_, K), dev), None, *wd,
                                   to_dev(offs, dev), N, K)
    torch.cuda.synchronize()
    assert_close(out.cpu().numpy(), ref, "mx gemm case %d" % case)


def test_mx_gemm_one_hot_exact(orc):
    """One-hot activation rows pick out weight columns: every product but one
    is zero, so the result is exact whatever the summation order."""
    dev = cuda_or_skip()
    E, N, K = 3, 256, 512
    W = np.stack([wl.expert_weight_fp32("w2", e, N, K, 5).numpy() for e in range(E)])
    w = orc.mx_quantize_experts(W)
    picks = [(0, 3), (0, 255), (1, 0), (2, 511), (2, 64)]
    offs = np.array([0, 2, 3, 5], np.int32)
    a = np.zeros((5, K), np.float32)
    for i, (_, c) in enumerate(picks):
        a[i, c] = 1.0
    ac, as_ = orc.mx_quantize(a)
    wd = upload_mx_weights(w, E, N, K, dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_MXW4A4, to_dev(ac, dev), to_dev(pad_scales(as_, K), dev), None, *wd,
                                   to_dev(offs, dev), N, K).cpu().numpy()
    for i, (e, c) in enumerate(picks):
        col = orc.mx_dequantize(w[0][e], w[1][e], K)[:, c]
        assert np.array_equal(out[i].astype(np.float64), col), (e, c)


# ---------------------------------------------------------------------------
# SwiGLU + MXFP4 requantisation, fused front half
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("R,I", [(1, 32), (37, 512), (128, 2048)])
def test_mx_swiglu_requant(orc, R, I):
    dev = cuda_or_skip()
    G = wl.random_fp32((R, 2 * I), seed=R + 3 * I, scale=1.5, tag="G").numpy()
    hc, hs = B.moe_swiglu_requant(to_dev(G, dev), B.MOE_MXW4A4)
    torch.cuda.synchronize()
    h32 = orc.swiglu(G).astype(np.float32)
    oc, os_ = orc.mx_quantize(h32)
    amb = mx_ambiguous(h32)
    gs = hs.cpu().numpy()
    assert not gs[:, I // 32:].any()
    bad_scale = (gs[:, : I // 32] != os_) & ~amb.reshape(R, I // 32, 32).any(-1)
    bad_code = (unpack_codes(hc.cpu().numpy()) != unpack_codes(oc)) & ~amb
    assert not bad_scale.any() and not bad_code.any()


@pytest.mark.parametrize("name", ["tiny", "decode_c16", "decode_b512"])
def test_mx_route_quantize_fused_matches_staged(orc, name):
    dev = cuda_or_skip()
    cfg = wl.CONFIGS[name]
    logits = wl.router_logits(cfg, device=dev)
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    fused = B.moe_route_quantize_mxfp4(x, logits, cfg.k)
    codes, scales = B.mxfp4_quantize(x)
    staged = B.moe_align_permute(logits, cfg.k)
    torch.cuda.synchronize()
    for key in ("ids", "w", "offsets", "perm", "inv"):
        assert torch.equal(fused[key], staged[key]), key
    perm = staged["perm"].long()
    assert torch.equal(fused["act_codes"], codes[perm])
    assert torch.equal(fused["act_scales"], scales[perm])
    oc, os_ = orc.mx_quantize(x.float().cpu().numpy())
    assert np.array_equal(codes.cpu().numpy(), oc)


# ---------------------------------------------------------------------------
# layer
# ---------------------------------------------------------------------------

def _oracle_weights(orc, cfg, experts, device="cpu"):
    w13 = orc.mx_quantize_experts(np.stack([wl.expert_weight_fp32("w13", e, 2 * cfg.I, cfg.H, 0, device).cpu().numpy()
                                            for e in experts]))
    w2 = orc.mx_quantize_experts(np.stack([wl.expert_weight_fp32("w2", e, cfg.H, cfg.I, 0, device).cpu().numpy()
                                           for e in experts]))
    return w13, w2


def gpu_mx_weights(cfg, dev):
    """Quantise every expert with the library's MXFP4 quantiser, pack scales."""
    out = []
    for which, N, K in (("w13", 2 * cfg.I, cfg.H), ("w2", cfg.H, cfg.I)):
        codes = torch.empty(cfg.E, N, K // 2, dtype=torch.uint8, device=dev)
        lin = torch.empty(cfg.E, N, K // 32, dtype=torch.uint8, device=dev)
        for e in range(cfg.E):
            wf = wl.expert_weight_fp32(which, e, N, K, 0, device=dev)
            c, s = B.mxfp4_quantize(wf, codes=codes[e])
            lin[e].copy_(s[:, : K // 32])
        packed = B.mxfp4_pack_weight_scales(lin, cfg.E, N, K)
        out.append(((codes, packed, None), lin))
    return out


def staged_mx(x, logits, cfg, w13, w2):
    k, I, H = cfg.k, cfg.I, cfg.H
    rt = B.moe_route_quantize_mxfp4(x, logits, k)
    G = B.moe_grouped_gemm_nvfp4(B.MOE_MXW4A4, rt["act_codes"], rt["act_scales"], None, *w13, rt["offsets"],
                                 2 * I, H)
    hc, hs = B.moe_swiglu_requant(G, B.MOE_MXW4A4)
    Y = B.moe_grouped_gemm_nvfp4(B.MOE_MXW4A4, hc, hs, None, *w2, rt["offsets"], H, I)
    out = B.moe_combine(Y, rt["inv"], rt["w"])
    return dict(rt=rt, G=G, hc=hc, hs=hs, Y=Y, out=out)


def test_mx_layer_tiny_all_intermediates(orc):
    dev = cuda_or_skip()
    cfg = wl.CONFIGS["tiny"]
    xt = wl.activations_bf16(cfg.T, cfg.H)
    logits = wl.router_logits(cfg)
    w13, w2 = _oracle_weights(orc, cfg, range(cfg.E))
    ref, mids = orc.moe_layer("mxw4a4", xt.float().numpy(), logits.numpy(), cfg.k, w13, w2, 0.0, intermediates=True)
    g13 = upload_mx_weights(w13, cfg.E, 2 * cfg.I, cfg.H, dev)
    g2 = upload_mx_weights(w2, cfg.E, cfg.H, cfg.I, dev)
    x, lg = xt.to(dev), logits.to(dev)
    d = staged_mx(x, lg, cfg, g13, g2)
    fused = B.moe_layer_forward(B.MOE_MXW4A4, x, lg, cfg.k, g13, g2, None)
    torch.cuda.synchronize()
    assert torch.equal(fused, d["out"])
    assert np.array_equal(d["rt"]["ids"].cpu().numpy(), mids["ids"])
    assert np.array_equal(d["rt"]["offsets"].cpu().numpy(), mids["offsets"])
    assert np.array_equal(d["rt"]["inv"].cpu().numpy(), mids["inv"])
    amb = mx_ambiguous(mids["h32"], rel=FLIP_WINDOW)
    flips = unpack_codes(d["hc"].cpu().numpy()) != unpack_codes(mids["hq_codes"])
    assert not (flips & ~amb).any()
    assert_close(d["out"].cpu().numpy(), ref, "tiny mxw4a4")


@pytest.mark.parametrize("name", ["decode_c16", "wide"])
def test_mx_layer_full_size(orc, name):
    """Every token of the batch against the oracle (see layer_parity)."""
    dev = cuda_or_skip()
    cfg = wl.CONFIGS[name]
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    logits = wl.router_logits(cfg, device=dev)
    (g13, l13), (g2, l2) = gpu_mx_weights(cfg, dev)
    d = staged_mx(x, logits, cfg, g13, g2)
    fused = B.moe_layer_forward(B.MOE_MXW4A4, x, logits, cfg.k, g13, g2, None)
    torch.cuda.synchronize()
    assert torch.equal(fused, d["out"]), "moe_layer_forward differs from the staged calls"
    check_layer(orc, cfg, "mxw4a4", d, x, logits, ((g13[0], l13), (g2[0], l2)), device=dev)


def test_mx_layer_decode_b512_full_size(orc):
    """decode_b512 in MXFP4: 128 tokens spread over the batch (every fourth),
    against the oracle (see layer_parity)."""
    dev = cuda_or_skip()
    cfg = wl.CONFIGS["decode_b512"]
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    logits = wl.router_logits(cfg, device=dev)
    (g13, l13), (g2, l2) = gpu_mx_weights(cfg, dev)
    d = staged_mx(x, logits, cfg, g13, g2)
    fused = B.moe_layer_forward(B.MOE_MXW4A4, x, logits, cfg.k, g13, g2, None)
    torch.cuda.synchronize()
    assert torch.equal(fused, d["out"]), "moe_layer_forward differs from the staged calls"
    check_layer(orc, cfg, "mxw4a4", d, x, logits, ((g13[0], l13), (g2[0], l2)), tokens=np.arange(0, cfg.T, 4),
                device=dev)
