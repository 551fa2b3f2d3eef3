"""GPU parity of moe_swiglu_requant and moe_combine against the oracle."""
import numpy as np
import pytest
import torch

from gpu_helpers import assert_close, cuda_or_skip, nvfp4_ambiguous, to_dev, unpack_codes
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _G(R, I, seed, scale=1.5):
    return wl.random_fp32((R, 2 * I), seed=seed, scale=scale, tag="G").numpy()


@pytest.mark.parametrize("R,I", [(1, 16), (37, 512), (128, 2048)])
def test_swiglu_requant_w4a4(orc, R, I):
    """Codes and scales bit for bit, except where the oracle's own fp32 h
    sits within 1e-5 of a rounding midpoint (the GPU evaluates exp in fp32,
    the oracle in fp64, so the last bits of h may differ there)."""
    dev = cuda_or_skip()
    G = _G(R, I, seed=R + I)
    S_h = np.float32(16 * 1.5 ** 4 / 2688)
    hc, hs = B.moe_swiglu_requant(to_dev(G, dev), B.MOE_W4A4, to_dev(np.array([S_h]), dev))
    torch.cuda.synchronize()
    h32 = orc.swiglu(G).astype(np.float32)
    oc, os_, _ = orc.quantize(h32, S_h)
    gs = hs.cpu().numpy()
    gcodes = unpack_codes(hc.cpu().numpy())
    ocodes = unpack_codes(oc)
    amb = nvfp4_ambiguous(h32, S_h)
    bad_scale = (gs != os_) & ~amb.reshape(R, I // 16, 16).any(-1)
    bad_code = (gcodes != ocodes) & ~amb
    assert not bad_scale.any() and not bad_code.any()
    assert (gcodes != ocodes).mean() < 1e-3


@pytest.mark.parametrize("R,I", [(5, 64), (256, 2048)])
def test_swiglu_w4a16_bf16(orc, R, I):
    dev = cuda_or_skip()
    G = _G(R, I, seed=7 * R)
    hb = B.moe_swiglu_requant(to_dev(G, dev), B.MOE_W4A16)
    torch.cuda.synchronize()
    ref = orc.swiglu(G)
    got = hb.float().cpu().numpy()
    # bf16 rounding of the fp32 value: at most half a bf16 ulp (<= 2^-8
    # relative at the bottom of a binade) plus fp32 noise
    err = np.abs(got - ref)
    assert np.all(err <= np.abs(ref) * (2.0 ** -8 + 1e-6) + 1e-30)


@pytest.mark.parametrize("T,k,H", [(1, 1, 4), (16, 8, 4096), (64, 22, 256), (7, 3, 6144)])
def test_combine(orc, T, k, H):
    dev = cuda_or_skip()
    rng = np.random.default_rng(T * k)
    Y = rng.normal(0, 1, (T * k, H)).astype(np.float32)
    inv = rng.permutation(T * k).astype(np.int32)
    w = rng.dirichlet(np.ones(k), T).astype(np.float32)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_combine(to_dev(Y, dev), to_dev(inv, dev), to_dev(w, dev), dev_status=status)
    ref = orc.combine(Y, inv.reshape(T, k).ravel(), w.astype(np.float64))
    assert_close(out.cpu().numpy(), ref, "combine")
    assert int(status.item()) == 0
    outb = B.moe_combine(to_dev(Y, dev), to_dev(inv, dev), to_dev(w, dev), out_dtype=torch.bfloat16)
    assert np.allclose(outb.float().cpu().numpy(), ref, rtol=2 ** -8, atol=1e-6)


def test_combine_out_of_range_rows_report_status(orc):
    """moe_combine takes the permutation from the caller: an entry outside
    [0, T*k) (one past the end, negative, far out) is never read.  Its term is
    skipped, NVFP4_E_BAD_ROUTING is reported in the status word, and the
    in-range terms are still summed."""
    dev = cuda_or_skip()
    T, k, H = 4, 3, 256
    rng = np.random.default_rng(11)
    Y = rng.normal(0, 1, (T * k, H)).astype(np.float32)
    inv = rng.permutation(T * k).astype(np.int32)
    w = rng.dirichlet(np.ones(k), T).astype(np.float32)
    bad = inv.copy()
    bad_slots = (1, 5, 7)
    bad[1], bad[5], bad[7] = T * k, -1, 1 << 30
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = B.moe_combine(to_dev(Y, dev), to_dev(bad, dev), to_dev(w, dev), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 8  # NVFP4_E_BAD_ROUTING
    w_ref = w.astype(np.float64).ravel().copy()
    inv_ref = bad.copy()
    for i in bad_slots:  # a skipped term: weight 0 on an in-range row
        w_ref[i] = 0.0
        inv_ref[i] = 0
    ref = orc.combine(Y, inv_ref, w_ref.reshape(T, k))
    assert_close(out.cpu().numpy(), ref, "combine with skipped rows")
