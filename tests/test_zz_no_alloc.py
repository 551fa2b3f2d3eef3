"""moe_align_permute_noalloc: the routing entry point for callers that cannot
give the library scratch memory (a host that owns all device memory and offers
no workspace, or a latency-critical path that must not call cudaMalloc).

It is checked through the C ABI against the ordinary moe_align_permute (which
takes a caller workspace) on the same inputs: identical ids, offsets,
permutation and gathered rows, routing weights within 1e-6.  Several calls in
a row, each over the previous call's leftovers in the shared fixed scratch
(which is never cleared between calls): decode_b512 twice (16 routing chunks
of 32 tokens), then wide (2 chunks, 512 experts: its masks land on top of the
previous call's), then decode_c16 (one chunk).  decode_b512 is also compared
with the oracle directly.  A problem whose eight-token routing blocks would
not fit the fixed scratch (1500 tokens, 1024 experts) routes in blocks of 32
there and still matches.  The file is named so that pytest collects it last.
"""
import ctypes as C

import numpy as np
import pytest
import torch

from gpu_helpers import cuda_or_skip
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SCRATCH_LIMIT = 512 * 1024  # NVFP4MOE_NOALLOC_SCRATCH_BYTES


def _p(t):
    return None if t is None else C.c_void_p(t.data_ptr())


def _outputs(T, E, k, H, dev):
    R = T * k
    return dict(ids=torch.empty(T, k, dtype=torch.int32, device=dev), w=torch.empty(T, k, device=dev),
                offsets=torch.empty(E + 1, dtype=torch.int32, device=dev),
                perm=torch.empty(R, dtype=torch.int32, device=dev), inv=torch.empty(R, dtype=torch.int32, device=dev),
                codes=torch.empty(R, H // 2, dtype=torch.uint8, device=dev),
                scales=torch.empty(R, H // 16, dtype=torch.uint8, device=dev),
                status=torch.zeros(1, dtype=torch.int32, device=dev))


def _call(noalloc, logits, k, xc, xs, out):
    L = B.load()
    T, E = logits.shape
    H = xc.shape[1] * 2
    st = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    common = (_p(logits), T, E, k, _p(out["ids"]), _p(out["w"]), _p(out["offsets"]), _p(out["perm"]), _p(out["inv"]),
              B.MOE_ACT_NVFP4, _p(xc), _p(xs), H, _p(out["codes"]), _p(out["scales"]), _p(out["status"]))
    if noalloc:
        return L.moe_align_permute_noalloc(*common, st)
    ws = torch.empty(max(int(L.moe_align_permute_workspace_bytes(T, E, k)), 256), dtype=torch.uint8,
                     device=logits.device)
    return L.moe_align_permute(*common, _p(ws), ws.numel(), st)


def _case(name, dev):
    cfg = wl.CONFIGS[name]
    logits = wl.router_logits(cfg, device=dev)
    x = wl.activations_bf16(cfg.T, cfg.H, device=dev)
    xc, xs, _ = B.nvfp4_quantize(x)
    return cfg, logits, xc, xs


def test_noalloc_matches_workspace_entry_point_twice(orc):
    dev = cuda_or_skip()
    # multi-chunk problems first (they use the fixed scratch), each over the
    # previous call's leftovers, then a single-chunk one
    for name in ("decode_b512", "decode_b512", "wide", "decode_c16"):
        cfg, logits, xc, xs = _case(name, dev)
        ref = _outputs(cfg.T, cfg.E, cfg.k, cfg.H, dev)
        got = _outputs(cfg.T, cfg.E, cfg.k, cfg.H, dev)
        assert _call(False, logits, cfg.k, xc, xs, ref) == 0
        assert _call(True, logits, cfg.k, xc, xs, got) == 0
        torch.cuda.synchronize()
        for key in ("ids", "offsets", "perm", "inv", "codes", "scales", "status"):
            assert torch.equal(got[key], ref[key]), (name, key)
        assert torch.allclose(got["w"], ref["w"], rtol=1e-6, atol=0), name
        if name == "decode_b512":
            # and directly against the oracle: routing and permutation bit for bit
            ids, w = orc.route(logits.cpu().numpy(), cfg.k)
            offsets, perm, inv = orc.permute(ids, cfg.E)
            assert np.array_equal(got["ids"].cpu().numpy(), ids)
            assert np.array_equal(got["offsets"].cpu().numpy(), offsets)
            assert np.array_equal(got["perm"].cpu().numpy(), perm)
            assert np.array_equal(got["inv"].cpu().numpy(), inv)
            assert np.allclose(got["w"].cpu().numpy(), w, rtol=0, atol=1e-6)


def test_noalloc_refuses_problems_beyond_its_scratch():
    dev = cuda_or_skip()
    E, k = 1024, 8
    T = 4096 + 32  # 256 + 4 * ceil(T/32) * E = 256 + 4 * 129 * 1024 bytes > 512 KB
    assert 256 + 4 * ((T + 31) // 32) * E > SCRATCH_LIMIT
    logits = torch.zeros(T, E, device=dev)
    out = _outputs(T, E, k, 256, dev)
    xc = torch.zeros(T, 128, dtype=torch.uint8, device=dev)
    xs = torch.zeros(T, 16, dtype=torch.uint8, device=dev)
    assert _call(True, logits, k, xc, xs, out) == 4  # NVFP4_E_WORKSPACE, nothing launched


def test_noalloc_routes_in_32_token_blocks_when_the_scratch_is_short(orc):
    """T = 1500, E = 1024: moe_align_permute routes in blocks of eight tokens,
    whose masks (4 * 47 blocks * 1024 experts * 4 B) would not fit the fixed
    scratch; the no-allocation entry point falls back to blocks of 32 tokens
    (47 * 1024 * 4 B) and must give the same routing and rows."""
    dev = cuda_or_skip()
    T, E, k, H = 1500, 1024, 8, 256
    nb = (T + 31) // 32
    assert 256 + 4 * 4 * nb * E > SCRATCH_LIMIT and 256 + 4 * nb * E + 4 * nb + 512 <= SCRATCH_LIMIT
    cfg = wl.MoEConfig("noalloc_fallback", T=T, H=H, I=256, E=E, k=k, routing="uniform")
    logits = wl.router_logits(cfg, seed=9, device=dev)
    x = wl.activations_bf16(T, H, seed=9, device=dev)
    xc, xs, _ = B.nvfp4_quantize(x)
    ref = _outputs(T, E, k, H, dev)
    got = _outputs(T, E, k, H, dev)
    assert _call(False, logits, k, xc, xs, ref) == 0
    assert _call(True, logits, k, xc, xs, got) == 0
    torch.cuda.synchronize()
    for key in ("ids", "offsets", "perm", "inv", "codes", "scales", "status"):
        assert torch.equal(got[key], ref[key]), key
    assert torch.allclose(got["w"], ref["w"], rtol=1e-6, atol=0)
    ids, w = orc.route(logits.cpu().numpy(), k)
    offsets, perm, inv = orc.permute(ids, E)
    assert np.array_equal(got["perm"].cpu().numpy(), perm)
    assert np.array_equal(got["offsets"].cpu().numpy(), offsets)
