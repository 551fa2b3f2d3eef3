"""GPU parity of moe_router_logits (router scores on the tensor cores,
K split over the SMs, partials added in a fixed order) against the oracle's
fp64 sum, and the routing that consumes them.

Bound per element: |GPU - oracle| <= 1e-5 * sum_h |x_h * w_eh| (fp32
accumulation of exact bf16 products over up to 6144 terms), plus the
relative-Frobenius / max-over-RMS bounds of the other float tests."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, to_dev
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SHAPES = [  # (T, H, E)
    (8, 256, 8),        # tiny: 8 experts in a 128-row tile
    (16, 4096, 256),    # decode C=16
    (64, 4096, 512),    # wide
    (512, 6144, 256),   # 512-token batch: 4 token tiles
    (33, 192, 130),     # ragged: 2 expert tiles, 2 token groups, 3 K chunks
    (1, 64, 1),         # one token, one expert, one K chunk
    (200, 128, 64),     # more token tiles than K chunks
]


def _inputs(T, H, E, seed):
    x = wl.activations_bf16(T, H, seed=seed)
    w = wl.router_weight_bf16(E, H, seed=seed)
    return x, w


@pytest.mark.parametrize("T,H,E", SHAPES)
def test_router_logits_vs_oracle(orc, T, H, E):
    dev = cuda_or_skip()
    x, w = _inputs(T, H, E, seed=T + E)
    got = B.moe_router_logits(x.to(dev), w.to(dev))
    again = B.moe_router_logits(x.to(dev), w.to(dev))
    torch.cuda.synchronize()
    assert torch.equal(got, again), "not reproducible"
    xf, wf = x.float().numpy(), w.float().numpy()
    ref = orc.router_logits(xf, wf).astype(np.float64)
    g = got.cpu().numpy().astype(np.float64)
    absum = np.abs(xf).astype(np.float64) @ np.abs(wf).astype(np.float64).T
    assert np.all(np.abs(g - ref) <= 1e-5 * absum + 1e-30)
    assert_close(g, ref, "router logits %dx%dx%d" % (T, H, E))


@pytest.mark.parametrize("T,H,E,k", [(16, 4096, 256, 8), (64, 4096, 512, 22)])
def test_router_logits_feed_routing(orc, T, H, E, k):
    """GPU logits -> GPU routing gives the oracle's experts for every token
    whose k-th and (k+1)-th oracle logits are more than 1e-4 apart (closer
    pairs may swap with the last bits of the sum); the rest are valid top-k
    sets of the GPU's own logits."""
    dev = cuda_or_skip()
    x, w = _inputs(T, H, E, seed=7)
    logits = B.moe_router_logits(x.to(dev), w.to(dev))
    rt = B.moe_align_permute(logits, k)
    torch.cuda.synchronize()
    ref = orc.router_logits(x.float().numpy(), w.float().numpy())
    ids_o, _ = orc.route(ref, k)
    ids_g = rt["ids"].cpu().numpy()
    srt = -np.sort(-ref, axis=1)
    clear = (srt[:, k - 1] - srt[:, k]) > 1e-4
    assert clear.mean() > 0.9
    assert np.array_equal(ids_g[clear], ids_o[clear])
    lg = logits.cpu().numpy()
    for t in np.where(~clear)[0]:
        kth = -np.sort(-lg[t])[k - 1]
        assert np.all(lg[t, ids_g[t]] >= kth)


def test_router_logits_rejects_bad_shapes():
    dev = cuda_or_skip()
    x = torch.zeros(4, 100, dtype=torch.bfloat16, device=dev)
    w = torch.zeros(8, 100, dtype=torch.bfloat16, device=dev)
    with pytest.raises(B.Nvfp4Error):
        B.moe_router_logits(x, w)  # H % 64 != 0


ROUTE_SHAPES = [  # (T, H, E, k)
    (16, 4096, 256, 8),   # decode C=16: the fused router kernel
    (1, 1024, 64, 4),     # one token
    (32, 2048, 512, 22),  # a full routing chunk, wide-expert top-k
    (7, 256, 1024, 32),   # the largest E and k the call accepts
    (33, 1024, 256, 8),   # two chunks: router GEMM + reduce + routing kernel
    (64, 4096, 512, 22),  # wide
]


@pytest.mark.parametrize("T,H,E,k", ROUTE_SHAPES)
def test_router_route_fused_matches_staged_and_oracle(orc, T, H, E, k):
    """moe_router_route (router GEMM + fused fixed-order reduce, top-k and
    permutation at T <= 32) is bitwise moe_router_logits followed by
    moe_align_permute, twice in a row (the completion counter resets itself),
    and its routing of its own logits is the oracle's bit for bit."""
    dev = cuda_or_skip()
    x, w = _inputs(T, H, E, seed=3 * T + E)
    x, w = x.to(dev), w.to(dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    first = B.moe_router_route(x, w, k, dev_status=status)
    got = B.moe_router_route(x, w, k, dev_status=status)
    lg = B.moe_router_logits(x, w)
    rt = B.moe_align_permute(lg, k)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    for key in ("ids", "w", "offsets", "perm", "inv"):
        assert torch.equal(got[key], first[key]), key
        assert torch.equal(got[key], rt[key]), key
    assert torch.equal(got["logits"], lg)
    ids, wts = orc.route(got["logits"].cpu().numpy(), k)
    offs, perm, inv = orc.permute(ids, E)
    assert np.array_equal(got["ids"].cpu().numpy(), ids)
    assert np.array_equal(got["offsets"].cpu().numpy(), offs)
    assert np.array_equal(got["perm"].cpu().numpy(), perm)
    assert np.array_equal(got["inv"].cpu().numpy(), inv)
    assert np.allclose(got["w"].cpu().numpy(), wts, rtol=0, atol=1e-6)
    # without the logits output the routing is the same
    nolog = B.moe_router_route(x, w, k, want_logits=False)
    torch.cuda.synchronize()
    assert torch.equal(nolog["perm"], got["perm"]) and torch.equal(nolog["w"], got["w"])
