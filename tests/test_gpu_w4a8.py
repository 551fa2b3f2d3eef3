"""GPU parity of the W4A8 mode (FP8 E4M3 activations with one per-tensor
scale x NVFP4 weights; "Native FP4 Is Slower Than Emulated FP4", section 1)
against the oracle: the FP8 quantiser and the fused route + quantise front
half bit for bit, the grouped GEMM on ragged expert groups (F16 operands,
exact), SwiGLU + FP8 requantisation, and the layer (tiny with every
intermediate; decode_c16 and wide at full size, every token)."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev, upload_weights
from layer_parity import FLIP_WINDOW, check_layer, fp8_boundary_distance
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl
from test_gpu_gemm import CASES, _offsets, _weights
from test_gpu_layer import gpu_weights

pytestmark = pytest.mark.gpu


def _hard(rows, cols, seed):
    """Normal values over a wide range, exact E4M3 midpoints (times the
    scale), tiny values of both signs and a saturating element."""
    rng = np.random.default_rng(seed)
    x = (rng.standard_normal((rows, cols)) * np.exp2(rng.integers(-6, 6, (rows, 1)))).astype(np.float32)
    if cols >= 32:
        x[0, :8] = [-1e-30, 1e-30, 0.0, -0.0, 3.0, -3.0, 1e30 if rows > 1 else 5.0, 2.0 ** -20]
    return x


@pytest.mark.parametrize("rows,cols", [(1, 16), (3, 96), (37, 512), (128, 4096)])
@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("dynamic", [True, False])
def test_fp8_quantize_bit_exact(orc, rows, cols, dtype, dynamic):
    dev = cuda_or_skip()
    x = torch.from_numpy(_hard(rows, cols, rows * cols)).to(dtype)
    xf = x.float().numpy()
    if dynamic:
        codes, S = B.fp8_quantize(x.to(dev))
        ref, S_ref = orc.fp8_quantize(xf)
    else:
        S_in = np.float32(0.037)
        codes, S = B.fp8_quantize(x.to(dev), S=torch.tensor([S_in], device=dev))
        ref, S_ref = orc.fp8_quantize(xf, S=S_in)
    torch.cuda.synchronize()
    assert float(S.item()) == float(S_ref)
    assert np.array_equal(codes.cpu().numpy(), ref)


@pytest.mark.parametrize("name", ["tiny", "decode_c16", "decode_b512"])
def test_route_quantize_fp8_matches_staged(orc, name):
    """The fused front half equals fp8_quantize + a row gather, bit for bit,
    and its routing and scale are the oracle's."""
    dev = cuda_or_skip()
    cfg = wl.CONFIGS[name]
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    logits = wl.router_logits(cfg, device=dev)
    rt = B.moe_route_quantize_fp8(x, logits, cfg.k)
    codes, S = B.fp8_quantize(x)
    torch.cuda.synchronize()
    assert float(rt["S_x"].item()) == float(S.item())
    assert torch.equal(rt["act_codes"], codes[rt["perm"].long()])
    ids, _ = orc.route(logits.cpu().numpy(), cfg.k)
    offs, perm, inv = orc.permute(ids, cfg.E)
    assert np.array_equal(rt["ids"].cpu().numpy(), ids) and np.array_equal(rt["perm"].cpu().numpy(), perm)
    assert float(S.item()) == float(orc.fp8_tensor_scale(x.float().cpu().numpy()))


def _codes_as_f16(codes):
    """FP8 E4M3 codes -> their values as float16 (every E4M3 value is one)."""
    return codes.view(torch.float8_e4m3fn).to(torch.float16)


@pytest.mark.parametrize("name", ["tiny", "decode_c16", "wide"])
def test_route_quantize_fp8_f16_carries_the_codes(orc, name):
    """The F16 carrier of the FP8 front half (what the W4A8 layer runs): the
    same routing and scale as moe_route_quantize_fp8, every code replaced by
    its value in f16, and the scale beside every row."""
    dev = cuda_or_skip()
    cfg = wl.CONFIGS[name]
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    logits = wl.router_logits(cfg, device=dev)
    rt = B.moe_route_quantize_fp8(x, logits, cfg.k)
    rf = B.moe_route_quantize_fp8_f16(x, logits, cfg.k)
    torch.cuda.synchronize()
    for key in ("ids", "offsets", "perm", "inv", "S_x"):
        assert torch.equal(rf[key], rt[key]), key
    assert torch.equal(rf["act_f16"].view(torch.int16), _codes_as_f16(rt["act_codes"]).view(torch.int16))
    assert torch.equal(rf["act_rs"], rt["S_x"].expand(rf["act_rs"].shape[0]))


@pytest.mark.parametrize("R,I", [(1, 16), (37, 512)])
def test_swiglu_fp8_f16_carries_the_codes(R, I):
    dev = cuda_or_skip()
    G = (wl.random_fp32((R, 2 * I), seed=R + I, tag="g8f") * 2).to(dev)
    S_h = torch.tensor([0.01], dtype=torch.float32, device=dev)
    hc = B.moe_swiglu_requant(G, B.MOE_W4A8, S_h=S_h)
    hf, rs = B.moe_swiglu_fp8_f16(G, S_h)
    torch.cuda.synchronize()
    assert torch.equal(hf.view(torch.int16), _codes_as_f16(hc).view(torch.int16))
    assert torch.equal(rs, S_h.expand(R))


def _fp8_acts(orc, R, K, seed):
    a = wl.random_fp32((R, K), seed=seed, tag="acts8").to(torch.bfloat16).float().numpy()
    return orc.fp8_quantize(a)


@pytest.mark.parametrize("case", range(len(CASES)))
def test_gemm_w4a8_ragged(orc, case):
    dev = cuda_or_skip()
    counts, N, K = CASES[case]
    E = len(counts)
    offs = _offsets(counts)
    R = int(offs[-1])
    w = _weights(orc, E, N, K, seed=case)
    ac, aS = _fp8_acts(orc, R, K, seed=500 + case)
    ref = orc.grouped_gemm_w4a8(ac, aS, w[0], w[1], w[2], offs)
    wd = upload_weights(w, E, N, K, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A8, to_dev(ac, dev), None, to_dev(np.array([aS]), dev), *wd,
                                   to_dev(offs, dev), N, K, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_close(out.cpu().numpy(), ref, "w4a8 case %d" % case)


def test_gemm_w4a8_one_hot_exact(orc):
    """Rows holding a single FP8 1.0 (code 0x38) pick out decoded weight
    columns times a_S * w_S exactly, whatever the summation order."""
    dev = cuda_or_skip()
    E, N, K = 2, 128, 512
    w = _weights(orc, E, N, K, seed=9)
    cols = [0, 1, 255, 256, 300, 511]
    ac = np.zeros((len(cols), K), np.uint8)
    for r, c in enumerate(cols):
        ac[r, c] = 0x38
    offs = _offsets([3, 3])
    ref = orc.grouped_gemm_w4a8(ac, np.float32(0.5), w[0], w[1], w[2], offs)
    wd = upload_weights(w, E, N, K, dev)
    out = B.moe_grouped_gemm_nvfp4(B.MOE_W4A8, to_dev(ac, dev), None, to_dev(np.array([0.5], np.float32), dev), *wd,
                                   to_dev(offs, dev), N, K)
    assert np.array_equal(out.cpu().numpy(), ref.astype(np.float32))


@pytest.mark.parametrize("R,I", [(1, 16), (37, 512), (128, 2048)])
def test_swiglu_requant_fp8(orc, R, I):
    """h = silu(g) * u requantised to FP8 with a static scale: codes equal the
    oracle's except where the oracle's fp32 h lies within FLIP_WINDOW of an
    E4M3 midpoint (the GPU evaluates exp in fp32)."""
    dev = cuda_or_skip()
    G = (wl.random_fp32((R, 2 * I), seed=R * 3 + I, tag="g8") * 2).numpy()
    S_h = np.float32(0.01)
    hc = B.moe_swiglu_requant(to_dev(G, dev), B.MOE_W4A8, S_h=to_dev(np.array([S_h]), dev))
    torch.cuda.synchronize()
    h32 = orc.swiglu(G).astype(np.float32)
    ref, _ = orc.fp8_quantize(h32, S=S_h)
    diff = hc.cpu().numpy() != ref
    assert not (diff & (fp8_boundary_distance(h32, S_h) > FLIP_WINDOW)).any()
    assert diff.mean() < 1e-3


def test_layer_w4a8_tiny_all_intermediates(orc):
    dev = cuda_or_skip()
    cfg = wl.CONFIGS["tiny"]
    xt = wl.activations_bf16(cfg.T, cfg.H)
    logits = wl.router_logits(cfg)
    w13 = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w13", e, 2 * cfg.I, cfg.H).numpy()
                                         for e in range(cfg.E)]))
    w2 = orc.quantize_experts(np.stack([wl.expert_weight_fp32("w2", e, cfg.H, cfg.I).numpy() for e in range(cfg.E)]))
    ref, mids = orc.moe_layer("w4a8", xt.float().numpy(), logits.numpy(), cfg.k, w13, w2, cfg.S_h8,
                              intermediates=True)
    g13 = upload_weights(w13, cfg.E, 2 * cfg.I, cfg.H, dev)
    g2 = upload_weights(w2, cfg.E, cfg.H, cfg.I, dev)
    S_h = torch.tensor([cfg.S_h8], dtype=torch.float32, device=dev)
    x, lg = xt.to(dev), logits.to(dev)
    d = staged_w4a8(x, lg, cfg, g13, g2, S_h)
    fused = B.moe_layer_forward(B.MOE_W4A8, x, lg, cfg.k, g13, g2, S_h)
    torch.cuda.synchronize()
    assert torch.equal(fused, d["out"])
    assert float(d["S_x"].item()) == float(mids["S_x"])
    assert np.array_equal(d["rt"]["inv"].cpu().numpy(), mids["inv"])
    flips = d["hc"].cpu().numpy() != mids["hq_codes"]
    assert not (flips & (fp8_boundary_distance(mids["h32"], cfg.S_h8) > FLIP_WINDOW)).any()
    assert_close(d["out"].cpu().numpy(), ref, "tiny w4a8")


def staged_w4a8(x, logits, cfg, w13, w2, S_h):
    k, I, H = cfg.k, cfg.I, cfg.H
    rt = B.moe_route_quantize_fp8(x, logits, k)
    G = B.moe_grouped_gemm_nvfp4(B.MOE_W4A8, rt["act_codes"], None, rt["S_x"], *w13, rt["offsets"], 2 * I, H)
    hc = B.moe_swiglu_requant(G, B.MOE_W4A8, S_h)
    Y = B.moe_grouped_gemm_nvfp4(B.MOE_W4A8, hc, None, S_h, *w2, rt["offsets"], H, I)
    out = B.moe_combine(Y, rt["inv"], rt["w"])
    return dict(rt=rt, S_x=rt["S_x"], G=G, hc=hc, Y=Y, out=out)


@pytest.mark.parametrize("name", ["decode_c16", "wide"])
def test_layer_w4a8_full_size(orc, name):
    """Every token of the batch against the oracle (see layer_parity)."""
    dev = cuda_or_skip()
    cfg = wl.CONFIGS[name]
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    logits = wl.router_logits(cfg, device=dev)
    (g13, s13), (g2, s2) = gpu_weights(cfg, dev)
    S_h = torch.tensor([cfg.S_h8], dtype=torch.float32, device=dev)
    d = staged_w4a8(x, logits, cfg, g13, g2, S_h)
    fused = B.moe_layer_forward(B.MOE_W4A8, x, logits, cfg.k, g13, g2, S_h)
    torch.cuda.synchronize()
    assert torch.equal(fused, d["out"]), "moe_layer_forward differs from the staged calls"
    check_layer(orc, cfg, "w4a8", d, x, logits, ((g13[0], s13), (g2[0], s2)), device=dev)
