"""GPU parity of nvfp4_quantize and nvfp4_pack_weight_scales against the
oracle: codes, scales and the dynamic per-tensor scale bit for bit."""
import numpy as np
import pytest
import torch

from gpu_helpers import cuda_or_skip, to_dev
from nvfp4_mixture_experts_top_gb300 import binding as B
from nvfp4_mixture_experts_top_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _run(orc, x_t, S=None):
    """GPU and oracle quantisation of the same input."""
    codes, scales, S_g = B.nvfp4_quantize(x_t, None if S is None else torch.tensor([S], dtype=torch.float32,
                                                                                     device=x_t.device))
    torch.cuda.synchronize()
    x_np = x_t.float().cpu().numpy()
    oc, os_, oS = orc.quantize(x_np, S)
    return (codes.cpu().numpy(), scales.cpu().numpy(), np.float32(S_g.cpu().numpy()[0])), (oc, os_, oS)


@pytest.mark.parametrize("shape", [(1, 16), (7, 48), (33, 256), (130, 1024)])
def test_quantize_bf16_dynamic(orc, shape):
    dev = cuda_or_skip()
    x = wl.random_fp32(shape, seed=shape[0], tag="q").to(torch.bfloat16).to(dev)
    (gc, gs, gS), (oc, os_, oS) = _run(orc, x)
    assert gS.view(np.uint32) == oS.view(np.uint32)
    assert np.array_equal(gs, os_)
    assert np.array_equal(gc, oc)


def test_quantize_full_decode_batch_activations(orc):
    """x [512, 6144] of the 512-token decode workload."""
    dev = cuda_or_skip()
    x = wl.activations_bf16(512, 6144, seed=0, device=dev)
    (gc, gs, gS), (oc, os_, oS) = _run(orc, x)
    assert gS == oS and np.array_equal(gs, os_) and np.array_equal(gc, oc)


def test_quantize_fp32_expert_weight(orc):
    """One gate_up weight matrix of the C=16 workload, fp32 input."""
    dev = cuda_or_skip()
    w = wl.expert_weight_fp32("w13", 3, 4096, 4096, seed=0, device=dev)
    (gc, gs, gS), (oc, os_, oS) = _run(orc, w)
    assert gS == oS and np.array_equal(gs, os_) and np.array_equal(gc, oc)


def test_quantize_static_scale_and_edge_values(orc):
    dev = cuda_or_skip()
    rng = np.random.default_rng(11)
    x = (rng.normal(0, 1, (64, 512)) * np.exp(rng.normal(0, 3, (64, 1)))).astype(np.float32)
    x[0, :16] = 0.0                                   # zero block
    x[1, :16] = -0.0                                  # negative zeros
    x[2, 3] = -1e-30                                  # rounds to -0
    x[3, :16] = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0, -0.25, -0.75, -1.25, -1.75, -2.5, -3.5, -5.0, -6.0]
    x[4, :16] = 1e30                                  # saturates the block scale
    x[5, 16:32] = np.float32(2.0 ** -126)             # denormal-scale region
    xt = to_dev(x, dev)
    for S in [1.0, 1.0 / 2688, 3.7e-4, 0.0, 1e-20]:
        (gc, gs, _), (oc, os_, _) = _run(orc, xt, S=S)
        assert np.array_equal(gs, os_), S
        assert np.array_equal(gc, oc), S


def test_quantize_dynamic_all_zero(orc):
    dev = cuda_or_skip()
    x = torch.zeros(3, 64, dtype=torch.bfloat16, device=dev)
    (gc, gs, gS), (oc, os_, oS) = _run(orc, x)
    assert gS == 0.0 and oS == 0.0 and not gc.any() and not gs.any()


def test_pack_weight_scales_layout():
    """Packed byte of (e, n, k-block j of 64-column block kb) sits at
    ((e*N/128 + n/128)*K/64 + kb)*512 + (n%32)*16 + ((n%128)/32)*4 + j."""
    dev = cuda_or_skip()
    E, N, K = 3, 256, 512
    rng = np.random.default_rng(12)
    lin = rng.integers(0, 256, (E, N, K // 16)).astype(np.uint8)
    packed = B.nvfp4_pack_weight_scales(to_dev(lin, dev), E, N, K).cpu().numpy()
    ref = np.zeros(E * N * K // 16, np.uint8)
    for e in range(E):
        for n in range(N):
            for kb in range(K // 64):
                for j in range(4):
                    off = ((e * (N // 128) + n // 128) * (K // 64) + kb) * 512 + (n % 32) * 16 + ((n % 128) // 32) * 4 + j
                    ref[off] = lin[e, n, kb * 4 + j]
    assert np.array_equal(packed, ref)
