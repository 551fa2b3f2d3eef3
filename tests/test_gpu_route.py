"""GPU parity of moe_align_permute against the oracle: expert ids, offsets,
permutation and inverse bit for bit; routing weights within 1e-6 relative;
the gathered activation rows byte for byte."""
import numpy as np
import pytest
import torch

from gpu_helpers import cuda_or_skip, to_dev
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _check(orc, logits_np, k, dev):
    out = B.moe_align_permute(to_dev(logits_np, dev), k)
    torch.cuda.synchronize()
    E = logits_np.shape[1]
    ids, w = orc.route(logits_np, k)
    offs, perm, inv = orc.permute(ids, E)
    assert np.array_equal(out["ids"].cpu().numpy(), ids)
    gw = out["w"].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(gw - w) <= 1e-6 * np.abs(w) + 1e-12)
    assert np.all(np.abs(gw.sum(1) - 1.0) <= 1e-6)
    assert np.array_equal(out["offsets"].cpu().numpy(), offs)
    assert np.array_equal(out["perm"].cpu().numpy(), perm)
    assert np.array_equal(out["inv"].cpu().numpy(), inv)
    return out


@pytest.mark.parametrize("name", ["tiny", "decode_c16", "decode_b512", "wide"])
def test_route_workloads(orc, name):
    dev = cuda_or_skip()
    cfg = wl.CONFIGS[name]
    _check(orc, wl.router_logits(cfg).numpy(), cfg.k, dev)


# 33..2432 tokens route in blocks of eight tokens (four per 32-token chunk);
# 2432 and 2433 sit on either side of that switch
@pytest.mark.parametrize("T,E,k", [(1, 8, 1), (33, 64, 8), (65, 1024, 32), (100, 7, 7), (31, 40, 3),
                                   (2432, 128, 8), (2433, 96, 4)])
def test_route_ragged_shapes(orc, T, E, k):
    dev = cuda_or_skip()
    logits = wl.random_fp32((T, E), seed=T * 1000 + E, tag="logits").numpy()
    _check(orc, logits, k, dev)


def test_route_ties_go_to_lower_id(orc):
    dev = cuda_or_skip()
    rng = np.random.default_rng(5)
    logits = rng.normal(0, 1, (40, 48)).astype(np.float32)
    logits[:, 10] = logits[:, 40]
    logits[:, 3] = logits[:, 33]
    logits[7, :] = 1.5
    logits[8, ::2] = 2.0
    _check(orc, logits, 6, dev)


def test_route_gather_nvfp4_and_bf16(orc):
    dev = cuda_or_skip()
    cfg = wl.CONFIGS["decode_c16"]
    logits = wl.router_logits(cfg).numpy()
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    codes, scales, _ = B.nvfp4_quantize(x)
    out = B.moe_align_permute(to_dev(logits, dev), cfg.k, act=(codes, scales), act_kind=B.MOE_ACT_NVFP4)
    perm = out["perm"].long()
    assert torch.equal(out["act_codes"], codes[perm])
    assert torch.equal(out["act_scales"], scales[perm])
    out = B.moe_align_permute(to_dev(logits, dev), cfg.k, act=x, act_kind=B.MOE_ACT_BF16)
    assert torch.equal(out["act_bf16"], x[out["perm"].long()])


def test_route_zero_tokens():
    dev = cuda_or_skip()
    out = B.moe_align_permute(torch.zeros(0, 16, device=dev), 2)
    assert not out["offsets"].cpu().numpy().any()


@pytest.mark.parametrize("name", ["tiny", "decode_c16", "decode_b512", "wide"])
def test_route_quantize_fused_matches_staged(orc, name):
    """moe_route_quantize_nvfp4 (routing + quantisation straight into
    permuted rows) gives exactly what nvfp4_quantize followed by
    moe_align_permute's NVFP4 gather gives, and the oracle's S_x."""
    dev = cuda_or_skip()
    cfg = wl.CONFIGS[name]
    logits = wl.router_logits(cfg, device=dev)
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    fused = B.moe_route_quantize_nvfp4(x, logits, cfg.k)
    codes, scales, S = B.nvfp4_quantize(x)
    staged = B.moe_align_permute(logits, cfg.k, act=(codes, scales), act_kind=B.MOE_ACT_NVFP4)
    torch.cuda.synchronize()
    for key in ("ids", "w", "offsets", "perm", "inv", "act_codes", "act_scales"):
        assert torch.equal(fused[key], staged[key]), key
    assert torch.equal(fused["S_x"], S)
    assert float(S.item()) == float(orc.tensor_scale(x.float().cpu().numpy()))
